"""Seeded synthetic inputs for the tree-verification hot path.

This module only draws random numbers and names fixed tree shapes. It holds none
of the method's arithmetic (no softmax, no top-k, no masks, no attention), so the
oracle side and the CUDA side can both take their inputs from it without sharing
any of the computation they are compared on.

Every draw comes from its own numpy PCG64 stream, keyed by (workload seed, what is
drawn, request, level), so a piece of input never depends on the order in which
the others were generated.

Shapes follow the five workloads of the tree-verification study:

  tiny      B=1, P=32, the fixed [2,2,1] tree of the handbook page's diagram
            (11 nodes), Hq=4, Hkv=2, D=64, fp32, q/k/v/cache ~ N(0,1), theta 1e4,
            draft and target tokens uniform over a vocabulary of 1000.
  llama8b   B=1, P=2048, Hq=32, Hkv=8, D=128, bf16 ~ N(0,1)/sqrt(128); dynamic
            tree with top_k=10, depth=6, total_tokens=60 from fp32 draft logits
            [10, 32000] per level ~ N(0, sigma=2).
  serving   the llama8b heads at B=16, P_b ~ U[512, 8192], KV in paged blocks of
            64 tokens behind a random block table; one 61-node tree per request.
  long70b   B=4, P=32768, Hq=64, Hkv=8, D=128, bf16; top_k=8, depth=7,
            total_tokens=48.
  sweep     B=64, P=1024, Hq=32, Hkv=8, D=128, bf16, total_tokens in
            {8, 16, 32, 64}; top_k=10, depth=6; draft logits [640, 128256].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# Parents of the handbook page's [2,2,1] diagram (root; A1, B1; A2, A2', B2, B2';
# A3, A3', B3, B3'), numbered breadth-first the way its build_draft_tree appends
# nodes. This is input data (a tree shape), not a computation.
TREE_221_PARENTS = (-1, 0, 0, 1, 1, 2, 2, 3, 4, 5, 6)

# Parents of the six-node example printed on the handbook page.
TREE_SIX_NODE_PARENTS = (-1, 0, 0, 1, 1, 2)

KV_BLOCK = 64  # tokens per paged KV block

_STREAMS = {
    "logits": 1, "q": 2, "k_new": 3, "v_new": 4, "k_cache": 5, "v_cache": 6,
    "prefix": 7, "blocks": 8, "root": 9, "target": 10, "tokens": 11, "pad": 12,
    "lm_hidden": 13, "lm_weight": 14, "t_logits": 15, "uniform": 16, "d_logits": 17,
}

# (hidden size, vocabulary) of the target model whose lm_head gives the greedy token at
# every node: Llama-3-8B (4096 x 128256) for the 8B-shaped workloads, Llama-3-70B
# (8192 x 128256) for the 70B-shaped one; a small head for the tiny tree.
TARGET_LM_HEAD = {"tiny": (64, 1000), "llama8b": (4096, 128256), "serving": (4096, 128256),
                  "long70b": (8192, 128256), "sweep": (4096, 128256)}
LM_WEIGHT_BLOCK = 8192  # vocabulary rows per weight draw


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                 # "f32" or "bf16"
    prefix: tuple              # ("fixed", P) or ("uniform", lo, hi)
    vocab: int
    top_k: int = 0             # 0: fixed tree (no expansion)
    depth: int = 0             # loop iterations after the base layer
    total_tokens: int = 0      # draft nodes kept (tree has total_tokens + 1 nodes)
    paged: bool = False
    fixed_parents: Optional[tuple] = None
    accept_p: float = 0.7      # continue-probability of the planted accepted walk
    logit_sigma: float = 2.0
    value_scale: Optional[float] = None  # None -> 1/sqrt(head_dim) for bf16, 1 for f32
    theta: float = 10000.0
    seed: int = 0

    @property
    def num_nodes(self) -> int:
        if self.fixed_parents is not None:
            return len(self.fixed_parents)
        return self.total_tokens + 1

    @property
    def num_candidates(self) -> int:
        """Store size of the dynamic expansion: top_k + depth * top_k**2."""
        return self.top_k + self.depth * self.top_k * self.top_k

    @property
    def max_prefix(self) -> int:
        return self.prefix[1] if self.prefix[0] == "fixed" else self.prefix[2]

    @property
    def scale(self) -> float:
        if self.value_scale is not None:
            return self.value_scale
        return 1.0 / math.sqrt(self.head_dim) if self.dtype == "bf16" else 1.0

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 2, 64, "f32", ("fixed", 32), 1000,
                     fixed_parents=TREE_221_PARENTS),
    "llama8b": Workload("llama8b", 1, 32, 8, 128, "bf16", ("fixed", 2048), 32000,
                        top_k=10, depth=6, total_tokens=60),
    "serving": Workload("serving", 16, 32, 8, 128, "bf16", ("uniform", 512, 8192), 32000,
                        top_k=10, depth=6, total_tokens=60, paged=True),
    "long70b": Workload("long70b", 4, 64, 8, 128, "bf16", ("fixed", 32768), 32000,
                        top_k=8, depth=7, total_tokens=48),
    "sweep": Workload("sweep", 64, 32, 8, 128, "bf16", ("fixed", 1024), 128256,
                      top_k=10, depth=6, total_tokens=64),
}
SWEEP_TOTAL_TOKENS = (8, 16, 32, 64)


def rng(w: Workload, stream: str, *key: int) -> np.random.Generator:
    """Independent PCG64 stream for one piece of one workload's input."""
    return np.random.default_rng(np.random.SeedSequence([w.seed, _STREAMS[stream], *key]))


def prefix_lengths(w: Workload) -> np.ndarray:
    if w.prefix[0] == "fixed":
        return np.full(w.batch, w.prefix[1], dtype=np.int32)
    lo, hi = w.prefix[1], w.prefix[2]
    return rng(w, "prefix").integers(lo, hi + 1, size=w.batch).astype(np.int32)


def draft_logits(w: Workload, b: int, level: int) -> np.ndarray:
    """fp32 draft logits of one request at one expansion level, ~ N(0, sigma).

    Level 1 (the base layer) has one row; every later level has top_k rows,
    one per frontier node, in the frontier's selection order.
    """
    rows = 1 if level == 1 else w.top_k
    g = rng(w, "logits", b, level)
    x = g.standard_normal((rows, w.vocab), dtype=np.float32)
    return (x * np.float32(w.logit_sigma)).astype(np.float32)


def draft_logits_batch(w: Workload, level: int) -> np.ndarray:
    """[B, rows, V] fp32 logits of every request at one level."""
    return np.stack([draft_logits(w, b, level) for b in range(w.batch)])


def root_tokens(w: Workload) -> np.ndarray:
    return rng(w, "root").integers(0, w.vocab, size=w.batch).astype(np.int32)


def fixed_tree_tokens(w: Workload, b: int, parents) -> np.ndarray:
    """Uniform node tokens for a fixed-shape tree, distinct among siblings."""
    g = rng(w, "tokens", b)
    n = len(parents)
    tok = np.zeros(n, dtype=np.int32)
    tok[0] = g.integers(0, w.vocab)
    for i in range(1, n):
        taken = {int(tok[j]) for j in range(1, i) if parents[j] == parents[i]}
        t = int(g.integers(0, w.vocab))
        while t in taken:
            t = int(g.integers(0, w.vocab))
        tok[i] = t
    return tok


def plant_target(w: Workload, b: int, tokens, parents, mode: str = "walk") -> np.ndarray:
    """Synthetic target argmax per node.

    mode "walk": every node's argmax is uniform over the vocabulary, then a walk
    from the root continues with probability accept_p into a uniformly chosen
    child, whose token becomes the current node's argmax; where the walk stops,
    the node's argmax is redrawn until it matches none of its children.
    mode "first": uniform argmax, except that the root's argmax is the token of
    node 1, so at least one draft token is accepted.
    """
    g = rng(w, "target", b)
    n = len(tokens)
    tgt = g.integers(0, w.vocab, size=n).astype(np.int32)
    if mode == "first":
        tgt[0] = tokens[1]
        return tgt
    node = 0
    while True:
        kids = [j for j in range(n) if parents[j] == node]
        if kids and g.random() < w.accept_p:
            c = kids[int(g.integers(0, len(kids)))]
            tgt[node] = tokens[c]
            node = c
            continue
        kid_tokens = {int(tokens[j]) for j in kids}
        t = int(g.integers(0, w.vocab))
        while t in kid_tokens:
            t = int(g.integers(0, w.vocab))
        tgt[node] = t
        return tgt


def normal(w: Workload, stream: str, shape, *key: int) -> np.ndarray:
    g = rng(w, stream, *key)
    return (g.standard_normal(shape, dtype=np.float32) * np.float32(w.scale)).astype(np.float32)


def new_qkv(w: Workload, t_max: Optional[int] = None):
    """q [B,T,Hq,D], k_new and v_new [B,T,Hkv,D], fp32 draws (to be cast to w.dtype)."""
    t = t_max or w.num_nodes
    q = normal(w, "q", (w.batch, t, w.num_q_heads, w.head_dim))
    k = normal(w, "k_new", (w.batch, t, w.num_kv_heads, w.head_dim))
    v = normal(w, "v_new", (w.batch, t, w.num_kv_heads, w.head_dim))
    return q, k, v


def prefix_kv(w: Workload, b: int, length: int):
    """Committed (already rotated) K and V of one request: [Hkv, length, D] each."""
    k = normal(w, "k_cache", (w.num_kv_heads, length, w.head_dim), b)
    v = normal(w, "v_cache", (w.num_kv_heads, length, w.head_dim), b)
    return k, v


def block_table(w: Workload, capacity_slots: int, pool_blocks: Optional[int] = None):
    """Random block table: request b's logical block j lives in physical block
    table[b, j]; the table is a prefix of a random permutation of the pool."""
    per_req = capacity_slots // KV_BLOCK
    need = w.batch * per_req
    pool = pool_blocks or need
    perm = rng(w, "blocks").permutation(pool).astype(np.int32)
    return perm[:need].reshape(w.batch, per_req), pool


def lm_head_hidden(w: Workload, rows: int, hidden: int, key: int = 0) -> np.ndarray:
    """[rows, hidden] fp32 draws ~ N(0, 1): the final-normed hidden state of every node
    (to be cast to bf16)."""
    return rng(w, "lm_hidden", key).standard_normal((rows, hidden), dtype=np.float32)


def lm_head_weight_blocks(w: Workload, vocab: int, hidden: int, key: int = 0):
    """The lm_head weight [vocab, hidden] ~ N(0, 1/sqrt(hidden)) as (v0, fp32 block) pairs
    of LM_WEIGHT_BLOCK rows, each from its own stream (to be cast to bf16)."""
    scale = np.float32(1.0 / math.sqrt(hidden))
    for j, v0 in enumerate(range(0, vocab, LM_WEIGHT_BLOCK)):
        n = min(LM_WEIGHT_BLOCK, vocab - v0)
        g = rng(w, "lm_weight", key, j)
        yield v0, (g.standard_normal((n, hidden), dtype=np.float32) * scale).astype(np.float32)


def target_logits(w: Workload, b: int, tokens, parents, vocab: int, t_max: int,
                  sigma: float = 2.0, boost: Optional[float] = None,
                  stream: str = "t_logits"):
    """[t_max, vocab] fp32 logits at every node of request b ~ N(0, sigma). Along a random
    root-down walk that continues with probability accept_p, the logit of the next node's
    token at its parent is raised by `boost` (default ln(vocab) + 4, which gives that
    token most of the mass at temperature 1, so probability tests pass often enough to
    walk the tree). Rows past the tree are drawn too."""
    if boost is None:
        boost = math.log(vocab) + 4.0
    g = rng(w, stream, b)
    x = (g.standard_normal((t_max, vocab), dtype=np.float32) * np.float32(sigma))
    n = len(parents)
    node = 0
    while True:
        kids = [c for c in range(n) if parents[c] == node]
        if not kids or g.random() >= w.accept_p:
            break
        c = kids[int(g.integers(0, len(kids)))]
        x[node, int(tokens[c])] += np.float32(boost)
        node = c
    return x.astype(np.float32)


def uniforms(w: Workload, b: int, n: int) -> np.ndarray:
    """n + 1 fp32 uniforms in [0, 1) of request b: one per node, then the final one."""
    return rng(w, "uniform", b).random(n + 1, dtype=np.float32)

"""One hot-path step over preallocated device buffers.

    draft expansion (depth + 1 levels) -> final selection -> tree metadata ->
    tree-verification attention (one layer) -> [target lm-head argmax per node] ->
    greedy acceptance + KV compaction

Every stage is one or two calls into libtsv.so on the current stream; no stage reads
anything back to the host, so a whole step can be captured in a CUDA graph.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

from . import _lib


@dataclasses.dataclass(frozen=True)
class TreeShape:
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    max_prefix: int
    vocab: int = 0
    top_k: int = 0
    depth: int = 0            # expansion loop iterations after the base layer
    total_tokens: int = 0     # draft nodes kept; the tree has total_tokens + 1 nodes
    fixed_nodes: int = 0      # > 0: trees are given directly (no expansion)
    fixed_max_depth: int = 0
    target_vocab: int = 0     # > 0: the target's lm_head runs in the step (its vocabulary)
    score_product: bool = False  # expansion scores as probability products, not log sums

    @property
    def max_nodes(self) -> int:
        return self.fixed_nodes if self.fixed_nodes else self.total_tokens + 1

    @property
    def max_depth(self) -> int:
        """Deepest node (edges from the root): one per draft level."""
        return self.fixed_max_depth if self.fixed_nodes else self.depth + 1

    @property
    def num_candidates(self) -> int:
        return self.top_k + self.depth * self.top_k * self.top_k


class HotPath:
    def __init__(self, shape: TreeShape, cache: _lib.KVCache, device=None):
        self.s = shape
        self.cache = cache
        dev = torch.device(device or cache.k.device)
        i32 = dict(dtype=torch.int32, device=dev)
        b, t, w = shape.batch, shape.max_nodes, (shape.max_nodes + 31) // 32
        if not shape.fixed_nodes:
            c, k = shape.num_candidates, shape.top_k
            self.store_token = torch.zeros(b, c, **i32)
            self.store_score = torch.zeros(b, c, dtype=torch.float32, device=dev)
            self.store_parent = torch.zeros(b, c, **i32)
            self.front = [(torch.zeros(b, k, **i32), torch.zeros(b, k, dtype=torch.float32, device=dev),
                           torch.zeros(b, k, **i32)) for _ in range(2)]
            ws = max(_lib.draft_topk_expand_workspace_size(b, 1, shape.vocab, k),
                     _lib.draft_topk_expand_workspace_size(b, k, shape.vocab, k))
            self.topk_ws = torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev)
        self.tokens = torch.full((b, t), -1, **i32)
        self.parents = torch.full((b, t), -1, **i32)
        self.num_nodes = torch.zeros(b, **i32)
        self.mask = torch.zeros(b, t, w, **i32)
        self.position_ids = torch.zeros(b, t, **i32)
        self.retrieve = torch.zeros(b, t, shape.max_depth + 1, **i32)
        self.num_leaves = torch.zeros(b, **i32)
        self.next_token = torch.zeros(b, t, **i32)
        self.next_sibling = torch.zeros(b, t, **i32)
        self.meta_err = torch.zeros(b, **i32)
        self.attn_err = torch.zeros(b, **i32)
        self.acc_err = torch.zeros(b, **i32)
        d = shape.head_dim
        self.out = torch.zeros(b, t, shape.num_q_heads, d, dtype=cache.dtype, device=dev)
        ws = _lib.tree_verify_attn_workspace_size((b, t, shape.num_q_heads, d), cache,
                                                  shape.max_prefix)
        if ws == 0:
            raise _lib.TsvError("tree_verify_attn rejects this shape")
        self.attn_ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.accept_path = torch.zeros(b, shape.max_depth + 1, **i32)
        self.accept_len = torch.zeros(b, **i32)
        self.bonus = torch.zeros(b, **i32)
        self.slot_map = torch.zeros(b, shape.max_depth + 1, 2, **i32)
        self.new_prefix_len = torch.zeros(b, **i32)
        self.sample_ws = torch.empty(max(_lib.tree_sample_accept_workspace_size(b, t), 256),
                                     dtype=torch.uint8, device=dev)
        if shape.target_vocab:
            self.target = torch.zeros(b, t, **i32)
            ws = _lib.lm_head_argmax_workspace_size(b * t, shape.target_vocab)
            self.lm_ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)

    # -- stages ------------------------------------------------------------------------
    def expand(self, level_logits: Sequence[torch.Tensor], root_token: torch.Tensor,
               level_ready: Optional[Sequence[torch.cuda.Event]] = None, select: bool = True):
        """level_logits[0]: [B, 1, V]; level_logits[l]: [B, K, V] fp32 (device).
        level_ready[l] (optional): an event after which level l's logits (and, for l = 0,
        root_token) are in place; the stream waits for it just before that level, so
        the logits of later levels can still be arriving while earlier levels run.
        select=False stops after the last level (select_tree then lays out the tree)."""
        s = self.s
        if len(level_logits) != s.depth + 1:
            raise ValueError(f"expected {s.depth + 1} levels of logits")
        cur = None
        for li, lg in enumerate(level_logits):
            if level_ready is not None and level_ready[li] is not None:
                torch.cuda.current_stream().wait_event(level_ready[li])
            nxt = self.front[li % 2]
            _lib.draft_topk_expand(lg, s.top_k, li + 1,
                                   None if cur is None else cur[1],
                                   None if cur is None else cur[2],
                                   self.store_token, self.store_score, self.store_parent,
                                   nxt[0], nxt[1], nxt[2], self.topk_ws,
                                   product=s.score_product)
            cur = nxt
        if select:
            _lib.draft_select_final(self.store_token, self.store_score, self.store_parent,
                                    s.num_candidates, s.total_tokens, root_token, self.tokens,
                                    self.parents, self.num_nodes)

    def select_tree(self, root_token: torch.Tensor, prefix_len: torch.Tensor):
        """The final selection and the selected trees' metadata in one launch (after
        expand(..., select=False)): the outputs of expand's selection and of build_meta."""
        s = self.s
        _lib.draft_select_tree(self.store_token, self.store_score, self.store_parent,
                               s.num_candidates, s.total_tokens, root_token, self.tokens,
                               self.parents, self.num_nodes, prefix_len, s.max_depth, self.mask,
                               self.position_ids, self.retrieve, self.num_leaves,
                               self.next_token, self.next_sibling, self.meta_err)

    def expand_fixed(self, level_logits: Sequence[torch.Tensor], root_token: torch.Tensor,
                     branching: Sequence[int]):
        """A fixed-branching tree instead of the dynamic expansion: level_logits[l] is
        [B, F_l, V] fp32 (F_l frontier nodes, the product of the earlier widths); the
        tree has 1 + sum over levels of F_l * branching[l] nodes (fixed_nodes)."""
        s = self.s
        n = 1
        frontier, first_parent = 1, 0
        self.tokens[:, 0].copy_(root_token)
        self.parents[:, 0] = -1
        for width, lg in zip(branching, level_logits):
            _lib.draft_fixed_level(lg, width, n, first_parent, self.tokens, self.parents)
            first_parent = n
            n += frontier * width
            frontier *= width
        if n != s.max_nodes:
            raise ValueError(f"branching {list(branching)} gives {n} nodes, max_nodes is "
                             f"{s.max_nodes}")
        self.num_nodes.fill_(n)

    def map_to_target(self, d2t: torch.Tensor, err: Optional[torch.Tensor] = None):
        """Draft-vocabulary ids of the tree's nodes (all but the root) to target ids."""
        _lib.draft_to_target(self.tokens, self.num_nodes, d2t, err)

    def set_tree(self, tokens: torch.Tensor, parents: torch.Tensor, num_nodes: torch.Tensor):
        """Use given trees instead of the expansion (fixed-shape drafts)."""
        self.tokens.copy_(tokens)
        self.parents.copy_(parents)
        self.num_nodes.copy_(num_nodes)

    def build_meta(self, prefix_len: torch.Tensor):
        _lib.tree_build_meta(self.parents, self.num_nodes, prefix_len, self.s.max_depth,
                             self.mask, self.position_ids, self.retrieve, self.num_leaves,
                             self.next_token, self.next_sibling, self.meta_err)

    def verify(self, q, k_new, v_new, prefix_len, rope_theta: float, softmax_scale: float):
        _lib.tree_verify_attn(q, k_new, v_new, self.cache, prefix_len, self.num_nodes,
                              self.position_ids, self.mask, rope_theta, softmax_scale, self.out,
                              self.attn_ws, self.s.max_prefix, self.attn_err)

    def greedy_targets(self, hidden: torch.Tensor, lm_weight: torch.Tensor):
        """The target's greedy token at every node: hidden [B, max_nodes, H] bf16 (the
        final-normed hidden state of each node), lm_weight [target_vocab, H] bf16 ->
        self.target [B, max_nodes] int32 (rows past a tree's num_nodes are computed too
        and never read by the walk)."""
        if not self.s.target_vocab:
            raise ValueError("TreeShape.target_vocab is 0: no lm_head stage")
        b, t = self.s.batch, self.s.max_nodes
        if hidden.dim() != 3 or hidden.shape[:2] != (b, t):
            raise ValueError(f"hidden must be [{b}, {t}, H]")
        if lm_weight.shape[0] != self.s.target_vocab:
            raise ValueError(f"lm_weight must have {self.s.target_vocab} rows")
        _lib.lm_head_argmax(hidden.view(b * t, hidden.shape[2]), lm_weight,
                            self.target.view(b * t), self.lm_ws)

    def accept(self, target_argmax, prefix_len, compact: bool = True, tree_valid=None):
        _lib.accept_and_compact(self.tokens, self.next_token, self.next_sibling, target_argmax,
                                self.num_nodes, prefix_len, self.s.max_depth,
                                self.cache if compact else None, self.accept_path,
                                self.accept_len, self.bonus, self.slot_map, self.new_prefix_len,
                                self.acc_err, tree_valid)

    def sample_accept(self, target_logits, temperature, top_k, top_p, min_p, u_node, u_final,
                      prefix_len, draft_probs=None, tree_valid=None, compact: bool = True):
        """Non-greedy acceptance of the current trees (tsv_tree_sample_accept): target
        logits [B, max_nodes, V] fp32, per-request sampling parameters [B], uniforms
        u_node [B, max_nodes] and u_final [B]; draft_probs [B, max_nodes, V] for the
        draft-aware rule (None: target-only). Writes the same outputs as accept()."""
        _lib.tree_sample_accept(target_logits, temperature, top_k, top_p, min_p, u_node, u_final,
                                self.tokens, self.next_token, self.next_sibling, self.num_nodes,
                                prefix_len, self.s.max_depth, self.cache if compact else None,
                                self.accept_path, self.accept_len, self.bonus, self.slot_map,
                                self.new_prefix_len, self.sample_ws, err=self.acc_err,
                                tree_valid=tree_valid, draft_probs=draft_probs)

    def step(self, level_logits, root_token, q, k_new, v_new, prefix_len, target_argmax,
             rope_theta: float, softmax_scale: float,
             level_ready: Optional[Sequence[torch.cuda.Event]] = None,
             inputs_ready: Optional[torch.cuda.Event] = None,
             hidden: Optional[torch.Tensor] = None, lm_weight: Optional[torch.Tensor] = None,
             sampling: Optional[dict] = None):
        """One hot-path step. level_ready (see expand) and inputs_ready (q, k_new, v_new,
        prefix_len and target_argmax or hidden in place before the tree metadata) let the
        inputs arrive on another stream while the expansion runs. With hidden and
        lm_weight (and target_argmax None) the target's greedy tokens come from the
        lm_head stage (greedy_targets) instead of being given. With `sampling` (the keyword
        arguments of sample_accept but prefix_len; target_argmax None) the acceptance is
        the non-greedy one."""
        if not self.s.fixed_nodes:
            self.expand(level_logits, root_token, level_ready, select=False)
        if inputs_ready is not None:
            torch.cuda.current_stream().wait_event(inputs_ready)
        if self.s.fixed_nodes:
            self.build_meta(prefix_len)
        else:
            self.select_tree(root_token, prefix_len)
        self.verify(q, k_new, v_new, prefix_len, rope_theta, softmax_scale)
        if sampling is not None:
            if target_argmax is not None or hidden is not None:
                raise ValueError("sampling replaces target_argmax / hidden")
            self.sample_accept(prefix_len=prefix_len, **sampling)
            return
        if hidden is not None:
            if target_argmax is not None:
                raise ValueError("give target_argmax or hidden + lm_weight, not both")
            self.greedy_targets(hidden, lm_weight)
            target_argmax = self.target
        self.accept(target_argmax, prefix_len)

    # launches of libtsv kernels per step (for the bench's launch count)
    def kernels_per_step(self, lm_head: bool = False) -> int:
        """libtsv kernels one step launches: one or two per expansion level (two for a
        large batch: streaming + merge), the final selection with the metadata (or the
        metadata alone for a fixed tree), the attention call, the lm_head stage (GEMM +
        finalize) when it runs, and the acceptance."""
        n = 0
        if not self.s.fixed_nodes:
            s = self.s
            n = sum(_lib.draft_topk_expand_launches(s.batch, 1 if lvl == 0 else s.top_k, s.vocab,
                                                    s.top_k) for lvl in range(s.depth + 1))
        return n + 1 + self.attn_kernels() + (2 if lm_head else 0) + 1

    def attn_kernels(self) -> int:
        """Kernels of one tree_verify_attn call: prep, the attention kernel (tensor-core
        for bf16 with head_dim 128 on sm_100 and later, CUDA-core otherwise) and the
        split merge when the keys are split."""
        return _lib.tree_verify_attn_launches(tuple(self.out.shape), self.cache, self.s.max_prefix)

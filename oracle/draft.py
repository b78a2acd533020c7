"""Draft-side dynamic tree expansion, oracle side (test infrastructure only).

[EAGLE2] section 3 (树的生长, topK_generate): a base layer takes the top_k tokens
of the root row; then, `depth` times, every one of the top_k frontier rows takes
its own top_k, each candidate's cumulative score is its parent's score plus its
log-probability (cu_scores = topk_p + scores[:, None]), and a joint top_k over
the top_k * top_k candidates gives the next frontier. All candidates are kept,
top_k + depth * top_k * top_k of them, and the total_tokens best are selected.

Candidate layout at a level: flat = s * K + c for frontier row s (in the previous
level's selection order) and the row's c-th best token, so the parent row of a
flat index is flat // K ([TRT] section 树的三套账, parents = topk_indices // K).

Ties, everywhere: higher value first, then the lower index (token id, flat index
or store index). [EAGLE2] section 5 breaks ties between paths by the lowest
index; the same rule is applied to every selection.

Precision: the log-sum-exp is taken in fp64; each log-probability is rounded once
to fp32 and the cumulative scores are fp32 sums, the precision in which the
selections are decided.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32


def logsumexp(row) -> float:
    """log(sum_v exp(x_v)) in fp64, shifted by the row maximum."""
    x = np.asarray(row, dtype=np.float64)
    m = float(x.max())
    return m + math.log(float(np.exp(x - m).sum()))


def log_softmax(row) -> np.ndarray:
    """fp64 log-probabilities of one row of logits."""
    x = np.asarray(row, dtype=np.float64)
    return x - logsumexp(x)


def row_topk(row, k: int) -> np.ndarray:
    """Token ids of the k largest logits, largest first, ties to the lower id.

    A full sort of the row by (value descending, id ascending); the first k.
    """
    x = np.asarray(row, dtype=np.float64)
    order = np.lexsort((np.arange(x.size), -x))  # last key is the primary key
    return order[:k].astype(np.int32)


def topk_by_score(scores, k: int) -> list:
    """Indices of the k highest fp32 scores, highest first, ties to the lower index."""
    s = [float(v) for v in np.asarray(scores, dtype=F32)]
    return sorted(range(len(s)), key=lambda i: (-s[i], i))[:k]


def selection_margin(scores, order_len: int) -> float:
    """Smallest gap between consecutive scores in the first order_len + 1 places of
    the descending order; how close a selection of order_len items came to a
    different outcome."""
    s = sorted((float(v) for v in np.asarray(scores, dtype=F32)), reverse=True)
    m = math.inf
    for a, b in zip(s[: order_len + 1], s[1: order_len + 1]):
        m = min(m, a - b)
    return m


class Level:
    """Result of one expansion level for one request."""

    def __init__(self, tokens, logp, cu, parent_store, selected):
        self.tokens = tokens            # int32 [R*K]  candidate token ids, flat order
        self.logp = logp                # fp32  [R*K]  log-probability of each candidate
        self.cu = cu                    # fp32  [R*K]  cumulative score
        self.parent_store = parent_store  # int32 [R*K] store index of the parent, -1 = root
        self.selected = selected        # list of K flat indices, best first


def expand_level(logits, k: int, parent_scores=None, parent_store=None,
                 product: bool = False) -> Level:
    """One topK_generate level ([EAGLE2] section 3).

    logits: [R, V] fp32, row s belongs to frontier node s (R = 1 at the base layer).
    parent_scores: fp32 [R] cumulative scores of the frontier (None: the root, 0; with
    product, 1).
    parent_store: int32 [R] store index of each frontier node (None: the root, -1).
    product: [TRT] section 树的三套账 (_select_topk_draft_tokens): the cumulative score is
    the parent's score times the child's probability (all_scores = new_scores *
    previous_scores), in probability form; the child's probability is exp of its fp32
    log-probability, rounded to fp32, and the product is an fp32 product.
    """
    logits = np.asarray(logits, dtype=F32)
    r = logits.shape[0]
    if parent_scores is None:
        parent_scores = (np.ones if product else np.zeros)(r, dtype=F32)
        parent_store = np.full(r, -1, dtype=np.int32)
    tokens = np.zeros(r * k, dtype=np.int32)
    logp = np.zeros(r * k, dtype=F32)
    cu = np.zeros(r * k, dtype=F32)
    pstore = np.zeros(r * k, dtype=np.int32)
    for s in range(r):
        lse = logsumexp(logits[s])
        top = row_topk(logits[s], k)
        for c in range(k):
            flat = s * k + c
            tokens[flat] = top[c]
            logp[flat] = F32(float(logits[s, top[c]]) - lse)
            if product:
                cu[flat] = F32(parent_scores[s]) * F32(math.exp(float(logp[flat])))
            else:
                cu[flat] = F32(parent_scores[s]) + logp[flat]  # fp32 sum
            pstore[flat] = parent_store[s]
    selected = topk_by_score(cu, k)
    return Level(tokens, logp, cu, pstore, selected)


def level_store_offset(level: int, k: int) -> int:
    """Store index of a level's first candidate: 0 for the base layer, then K, K+K^2, ..."""
    return 0 if level == 1 else k + (level - 2) * k * k


def num_candidates(k: int, depth: int) -> int:
    """top_k + depth * top_k * top_k ([EAGLE2] section 3; the page's '+' was lost in
    extraction); equal to [TRT]'s K + K^2 (D - 1) with D = depth + 1 levels."""
    return k + depth * k * k


class Expansion:
    def __init__(self, store_token, store_score, store_parent, levels):
        self.store_token = store_token
        self.store_score = store_score
        self.store_parent = store_parent
        self.levels = levels


def topk_generate(level_logits, k: int, product: bool = False) -> Expansion:
    """All levels of one request: level_logits[0] is [1, V], the rest [K, V]. product:
    the probability-product scores of expand_level."""
    depth = len(level_logits) - 1
    c = num_candidates(k, depth)
    store_token = np.zeros(c, dtype=np.int32)
    store_score = np.zeros(c, dtype=F32)
    store_parent = np.zeros(c, dtype=np.int32)
    levels = []
    front_scores = None
    front_store = None
    for li, lg in enumerate(level_logits):
        level = li + 1
        lv = expand_level(lg, k, front_scores, front_store, product)
        off = level_store_offset(level, k)
        n = lv.tokens.size
        store_token[off:off + n] = lv.tokens
        store_score[off:off + n] = lv.cu
        store_parent[off:off + n] = lv.parent_store
        front_scores = np.array([lv.cu[f] for f in lv.selected], dtype=F32)
        front_store = np.array([off + f for f in lv.selected], dtype=np.int32)
        levels.append(lv)
    return Expansion(store_token, store_score, store_parent, levels)


def select_final(store_token, store_score, store_parent, total_tokens: int, root_token: int):
    """Keep the total_tokens best candidates and lay them out as a tree.

    [EAGLE2] section 3: the total_tokens highest-scoring nodes are kept. They are
    numbered in ascending store index (so parents precede children), node 0 is the
    root, and each node's parent is mapped from its store index to its node index.
    Returns (tokens [T], parents [T]) with T = total_tokens + 1.
    """
    best = topk_by_score(store_score, total_tokens)
    chosen = sorted(best)
    node_of = {c: i + 1 for i, c in enumerate(chosen)}
    tokens = [int(root_token)] + [int(store_token[c]) for c in chosen]
    parents = [-1]
    for c in chosen:
        p = int(store_parent[c])
        if p < 0:
            parents.append(0)
        else:
            if p not in node_of:
                raise AssertionError("selected candidate whose parent was not selected")
            parents.append(node_of[p])
    return np.array(tokens, dtype=np.int32), np.array(parents, dtype=np.int32)


def margins(exp: Expansion, total_tokens: int) -> float:
    """Smallest decision gap over every joint top-k and the final selection."""
    m = math.inf
    k = len(exp.levels[0].selected)
    for lv in exp.levels:
        m = min(m, selection_margin(lv.cu, k))
    s = sorted((float(v) for v in exp.store_score), reverse=True)
    if total_tokens < len(s):
        m = min(m, s[total_tokens - 1] - s[total_tokens])
    return m


def map_draft_to_target(tokens, num_nodes: int, d2t):
    """Draft-vocabulary ids to target-vocabulary ids ([MO] section 独立小lm_head草稿词表压缩:
    the drafter predicts over a smaller vocabulary and a d2t buffer maps each draft id
    back, draft_token = d2t[draft_token]). Node 0 (the root, a token the target already
    committed) is left as it is; a draft id outside the table maps to -1, which no
    target token equals."""
    out = np.array(tokens, dtype=np.int32).copy()
    for i in range(1, num_nodes):
        t = int(out[i])
        out[i] = int(d2t[t]) if 0 <= t < len(d2t) else -1
    return out


def fixed_tree(level_logits, branching, root_token: int):
    """The fixed-shape draft tree of [HB] section 实现 (build_draft_tree): level l gives
    every frontier node its top-branching[l] tokens (larger logit first, lower id on
    ties), appended frontier node by frontier node. level_logits[l] is [F_l, V], row f
    the draft's logits at the l-th level's f-th frontier node. Returns (tokens, parents)."""
    tokens, parents, frontier = [int(root_token)], [-1], [0]
    for width, lg in zip(branching, level_logits):
        lg = np.asarray(lg, dtype=F32)
        assert lg.shape[0] == len(frontier)
        nxt = []
        for f, node in enumerate(frontier):
            for t in row_topk(lg[f], width):
                tokens.append(int(t))
                parents.append(node)
                nxt.append(len(tokens) - 1)
        frontier = nxt
    return np.array(tokens, dtype=np.int32), np.array(parents, dtype=np.int32)

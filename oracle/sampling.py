"""Non-greedy acceptance on the tree, oracle side (test infrastructure only).

[TRT] section 非贪心:只靠目标分布的拒绝采样: in the dynamic-tree mode the target's
logits at every node are filtered into probabilities with the request's sampling
parameters (temperature, top-k, top-p, min-p, each request's set repeated for each of
its nodes); the walk follows next_token / next_sibling and, instead of comparing a
child with the target's argmax, makes a probability test at each node, and where it
stops it samples a correction token from the target's distribution. Only the target's
logits are used (no draft probabilities are kept): "target-only" rejection.

[HB] section 练习, exercise 2 (采样时的树) and its reference answer: level by level, at a
node take its children (the draft's candidates) in turn; accept candidate x with
probability min(1, p(x) / q(x)); on a rejection replace the target distribution by
norm(max(0, p - q)) and go on to the next candidate; if every candidate is rejected,
sample one token from the last residual and stop. q is to be taken as the candidates
were drawn.

Readings (the pages leave these open; the plainest reading that the rest supports):
  * Target-only is the same rule with q = the point mass on the candidate being tested
    (the draft's token is treated as fixed): accept x with probability p(x); on a
    rejection p <- p with x removed, renormalised.
  * Draft-aware: q is one distribution per node, the one its children were drawn from,
    given by the caller. The siblings of a tree are distinct tokens, so they were drawn
    from q without replacement: the j-th candidate comes from q with the j - 1 tokens
    drawn before it removed and the rest renormalised. That is the q of each test and
    of each residual ("q as the candidates were drawn"): after a rejection of x the
    target side becomes norm(max(0, p - q)) with the q that x was tested against, and
    the draft side norm(q with q(x) = 0). If q has no mass left, the later candidates
    are tested against q = 0 (accepted wherever p > 0).
  * The filters apply in the order the page lists them: temperature, then top-k, then
    top-p on the renormalised result, then min-p on that. top-k keeps the k best
    logits (ties to the lower token id); top-p keeps, in that order, every token whose
    preceding mass is below top_p of the total (so the token that crosses is kept and
    at least one token always is); min-p keeps tokens whose probability is at least
    min(min_p, 1) times the largest one (the most likely token always stays).
    temperature 0 (or below, or NaN) is greedy: all mass on the first maximum; so are
    top_k = 1, top_p <= 0 and a row whose largest logit is not finite. NaN logits read
    as -inf.
  * An accepted child's node becomes the current node; when a node has no children,
    or all of them are rejected, one token is sampled from the current distribution
    (the residual after the rejections made at that node) and the walk ends. The
    sample is the inverse CDF in token-id order: the smallest t whose cumulative
    probability exceeds u.
  * The random numbers are inputs: u_node[c] is the uniform of the test of node c (a
    node is tested at most once, as a candidate of its parent) and u_final the uniform
    of the final sample, all in [0, 1).
"""
from __future__ import annotations

import numpy as np


def filter_probs(logits, temperature: float, top_k: int = 0, top_p: float = 1.0,
                 min_p: float = 0.0):
    """The filtered target distribution of one node (fp64 vector over the vocabulary).

    top_k <= 0 or >= V, top_p >= 1 and min_p <= 0 switch the filter off.
    """
    lg = np.asarray(logits, np.float64)
    lg = np.where(np.isnan(lg), -np.inf, lg)  # a NaN logit never wins
    v = lg.shape[0]
    if not temperature > 0.0 or top_k == 1 or top_p <= 0.0 or not np.isfinite(lg.max()):
        p = np.zeros(v)
        p[int(np.argmax(lg))] = 1.0  # the first maximum
        return p
    e = np.exp((lg - lg.max()) / temperature)
    order = np.lexsort((np.arange(v), -lg))  # larger logit first, then lower token id
    keep = np.ones(v, bool)
    if 0 < top_k < v:
        keep[:] = False
        keep[order[:top_k]] = True
    if top_p < 1.0:
        total = e[keep].sum()
        before, first = 0.0, True
        for t in order:
            if not keep[t]:
                continue
            if not first and before >= top_p * total:
                keep[t] = False
            before += e[t]
            first = False
    if min_p > 0.0:
        keep &= e >= min(min_p, 1.0) * e[keep].max()
    p = np.where(keep, e, 0.0)
    return p / p.sum()


def sample_inverse_cdf(p, u: float, trace=None) -> int:
    """The smallest token id t with sum(p[:t+1]) > u * sum(p). With a trace list, appends
    ("final", u, p): the distribution the token was drawn from."""
    c = np.cumsum(np.asarray(p, np.float64))
    t = min(int(np.searchsorted(c, u * c[-1], side="right")), len(c) - 1)
    if trace is not None:
        trace.append(("final", float(u), np.asarray(p, np.float64)))
    return t


def children(parents, node):
    return [c for c in range(len(parents)) if parents[c] == node]


def rejection_walk(tokens, parents, probs, u_node, u_final, q=None, tree_valid=True,
                   trace=None):
    """Tree rejection sampling for one request.

    tokens, parents: the tree (node 0 the root). probs[i]: the filtered target
    distribution at node i (filter_probs). q: None for target-only, else q[i] is the
    draft distribution the children of node i were drawn from, without replacement, in
    ascending node order. Returns (path, token):
    the accepted nodes from the root, and the token sampled where the walk stopped
    (the correction or bonus token). With a trace list, every test appends ("test", u,
    its acceptance probability) and the final sample ("final", u, the distribution), so
    a caller can see how far each decision was from flipping.
    """
    path, node = [0], 0
    if not tree_valid:
        return path, sample_inverse_cdf(probs[0], u_final, trace)
    while True:
        p = np.array(probs[node], np.float64)
        qc = None if q is None else np.array(q[node], np.float64)  # q of the next draw
        nxt = None
        for c in children(parents, node):
            x = int(tokens[c])
            qx = 1.0 if q is None else float(qc[x])
            ratio = np.inf if qx == 0.0 and p[x] > 0.0 else (0.0 if qx == 0.0 else p[x] / qx)
            if trace is not None:
                trace.append(("test", float(u_node[c]), min(1.0, ratio)))
            if u_node[c] < min(1.0, ratio):
                nxt = c
                break
            if q is None:
                resid = p.copy()
                resid[x] = 0.0
            else:
                resid = np.maximum(0.0, p - qc)
                # the next sibling was drawn from q without the tokens drawn before it
                qc[x] = 0.0
                sq = qc.sum()
                if sq > 0.0:
                    qc = qc / sq
            s = resid.sum()
            if s > 0.0:
                p = resid / s
        if nxt is None:
            return path, sample_inverse_cdf(p, u_final, trace)
        path.append(nxt)
        node = nxt

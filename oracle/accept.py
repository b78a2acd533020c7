"""Greedy acceptance and KV compaction, oracle side (test infrastructure only)."""
from __future__ import annotations

import numpy as np


def greedy_walk(tokens, parents, target, tree_valid=True):
    """Longest accepted root-down path, handbook form.

    [HB] section 实现 (tree_speculative_generate): start at the root; the target's
    argmax at the current node must equal the token of one of its children, the
    lowest-numbered such child is taken; stop when none matches. The bonus token is
    the target's argmax at the last accepted node. Returns (path, bonus); the path
    includes the root, so len(path) is the accepted length.

    [TRT] section 每请求一份树,按 slot 存放: a request whose tree is not valid (its slot
    was released: has_tree / tree_valid is false) takes the single-token path, so only
    the root is accepted.
    """
    n = len(tokens)
    path, node = [0], 0
    if not tree_valid:
        return path, int(target[0])
    for _ in range(n):
        pred = int(target[node])
        child = next((c for c in range(n) if parents[c] == node and tokens[c] == pred), None)
        if child is None:
            break
        path.append(child)
        node = child
    return path, int(target[node])


def evaluate_posterior(tokens, retrieve, target):
    """Best path by the EAGLE-2 rule ([EAGLE2] section 5, evaluate_posterior).

    For every retrieve row (root-to-leaf node indices, -1 padded) the draft at
    column i is accepted when it equals the target's argmax at column i-1; a
    cumulative product keeps only the leading run; the longest run wins, the lowest
    row on ties. Returns (row, accept_length) with accept_length counting accepted
    draft tokens (the root not included).
    """
    best_row, best_len = 0, -1
    for r, row in enumerate(retrieve):
        run = 1
        count = 0
        for i in range(1, len(row)):
            if row[i] < 0:
                break
            ok = 1 if int(tokens[row[i]]) == int(target[row[i - 1]]) else 0
            run *= ok
            count += run
        if count > best_len:
            best_row, best_len = r, count
    return best_row, best_len


def slot_map(prefix_len: int, path):
    """(source slot, destination slot) of every accepted node: the node's tree slot
    prefix_len + node moves to the sequence slot prefix_len + i."""
    return [(prefix_len + int(n), prefix_len + i) for i, n in enumerate(path)]


def compact(cache, prefix_len: int, path):
    """Move the accepted nodes' cache rows to consecutive slots ([HB] section 实现:
    only the path's KV is appended, nothing is recomputed; [TRT] section
    接受之后: KV 从树形搬回线性).

    cache: [..., S, D] array (any leading dims, slot axis second to last). The rows
    are read into a temporary first, so the result does not depend on copy order.
    Returns a new array.
    """
    out = np.array(cache, copy=True)
    src = [prefix_len + int(n) for n in path]
    tmp = np.array(out[..., src, :], copy=True)
    out[..., prefix_len:prefix_len + len(path), :] = tmp
    return out

"""Tree metadata, oracle side (test infrastructure only).

Nodes are numbered so that every parent precedes its children (node 0 is the
root, parents[0] == -1), as the handbook page's build_draft_tree appends them.
"""
from __future__ import annotations

import numpy as np


def validate_parents(parents) -> None:
    """Raise ValueError unless parents describes a rooted tree in parent-first order."""
    if len(parents) == 0 or parents[0] != -1:
        raise ValueError("node 0 must be the root (parent -1)")
    for i in range(1, len(parents)):
        if not (0 <= parents[i] < i):
            raise ValueError(f"parent of node {i} must lie in [0, {i})")


def tree_mask(parents) -> np.ndarray:
    """[T, T] bool: row i is True at i and at every ancestor of i.

    [HB] section 实现, tree_mask: walk from the node up to the root and mark each
    node met. [EAGLE2] section 3 calls the same matrix tree_mask[i][j].
    """
    n = len(parents)
    mask = np.zeros((n, n), dtype=bool)
    for i in range(n):
        j = i
        while j != -1:
            mask[i, j] = True
            j = parents[j]
    return mask


def depths(parents) -> list:
    """Root depth 0, every other node one deeper than its parent ([HB] 实现, depths)."""
    d = []
    for p in parents:
        d.append(0 if p == -1 else d[p] + 1)
    return d


def position_ids(parents, prefix_len: int) -> np.ndarray:
    """RoPE position of each node = committed prefix length + depth.

    [HB] section 为什么要用树 (siblings share a position) and 实现 (pos computed as
    len(committed) + depth); [EAGLE2] section 4 (tree_position_ids + input length).
    """
    return np.array([prefix_len + d for d in depths(parents)], dtype=np.int64)


def pack_mask(mask: np.ndarray, words: int | None = None) -> np.ndarray:
    """Bit-pack each mask row into uint32 words: column j -> word j//32, bit j%32.

    [TRT] section 树构建内核做了什么: 32 positions per int32 word (tree_mask_mode 2).
    The page does not fix the bit order; the lowest column goes to the least
    significant bit.
    """
    n, m = mask.shape
    w = words if words is not None else (m + 31) // 32
    out = np.zeros((n, w), dtype=np.uint32)
    for i in range(n):
        for j in range(m):
            if mask[i, j]:
                out[i, j // 32] |= np.uint32(1 << (j % 32))
    return out


def children_of(parents) -> list:
    kids = [[] for _ in parents]
    for i, p in enumerate(parents):
        if p >= 0:
            kids[p].append(i)
    return kids


def next_links(parents):
    """Child/sibling links ([TRT] 树构建内核做了什么: retrieve_next_token /
    retrieve_next_sibling, both -1 where absent).

    next_token[i]   = the lowest-numbered child of i, or -1.
    next_sibling[i] = the next higher-numbered child of parent(i), or -1.
    """
    n = len(parents)
    nxt = [-1] * n
    sib = [-1] * n
    kids = children_of(parents)
    for i in range(n):
        if kids[i]:
            nxt[i] = kids[i][0]
        for a, b in zip(kids[i], kids[i][1:]):
            sib[a] = b
    return np.array(nxt, dtype=np.int32), np.array(sib, dtype=np.int32)


def leaves(parents) -> list:
    kids = children_of(parents)
    return [i for i in range(len(parents)) if not kids[i]]


def retrieve_indices(parents, cols: int) -> np.ndarray:
    """[num_leaves, cols] int32: one row per leaf (leaves in ascending node order),
    the node indices on the root-to-leaf path, padded with -1.

    [EAGLE2] section 3: find the leaves, trace each back to the root, one row per
    path of shape [leaf_num, max_depth]. Padding value and leaf order are not fixed
    by the page; -1 and ascending node order are this oracle's reading.
    """
    rows = []
    for leaf in leaves(parents):
        path = []
        j = leaf
        while j != -1:
            path.append(j)
            j = parents[j]
        path.reverse()
        if len(path) > cols:
            raise ValueError("path longer than the retrieve_indices width")
        rows.append(path + [-1] * (cols - len(path)))
    return np.array(rows, dtype=np.int32).reshape(len(rows), cols)


def fixed_branching_parents(branching) -> list:
    """Parents of the tree that build_draft_tree grows ([HB] 实现): level l gives
    every frontier node branching[l] children, appended frontier node by node."""
    parents, frontier = [-1], [0]
    for width in branching:
        nxt = []
        for node in frontier:
            for _ in range(width):
                parents.append(node)
                nxt.append(len(parents) - 1)
        frontier = nxt
    return parents


def kary_parents(n: int, k: int) -> list:
    """Regular k-ary tree of n nodes: parent(i) = (i - 1) // k ([TRT] section
    dummy 槽为什么要造一棵 K 叉树; k = 1 gives the default linear chain)."""
    return [-1] + [(i - 1) // k for i in range(1, n)]


def grow_level_mask(prev_mask, prev_pos, new_parents):
    """The drafter's mask and positions after one more draft level, built as the block
    matrix of [TRT] section 首步变长、后续定长 (_build_mask_and_position): the old nodes keep
    their rows and see none of the new nodes (the upper-right block is zero); a new node's
    row is its parent's row (gathered from the old mask) followed by tree_mask_init, the
    new nodes' visibility among themselves (each sees itself only). A new node's position
    is its parent's plus one.

    prev_mask [N, N] bool, prev_pos [N], new_parents [K] (indices of old nodes).
    Returns ([N + K, N + K] bool, [N + K] positions)."""
    prev_mask = np.asarray(prev_mask, dtype=bool)
    n, k = prev_mask.shape[0], len(new_parents)
    parent_rows = prev_mask[np.asarray(new_parents, dtype=np.int64)]     # [K, N]
    top = np.concatenate([prev_mask, np.zeros((n, k), dtype=bool)], axis=1)
    bottom = np.concatenate([parent_rows, np.eye(k, dtype=bool)], axis=1)
    pos = np.concatenate([np.asarray(prev_pos, dtype=np.int64),
                          np.asarray(prev_pos, dtype=np.int64)[list(new_parents)] + 1])
    return np.concatenate([top, bottom], axis=0), pos

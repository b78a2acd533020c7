"""Tree-verification attention, oracle side (test infrastructure only).

[HB] section 实现, forward_with_mask: every tree node attends to the whole
committed prefix and, among the tree nodes, to itself and its ancestors; the mask
is materialised as [ones(T, P) | tree_mask] and applied to scaled dot-product
attention; grouped-query heads share a KV head by repeat_interleave. [HB] section
为什么要用树: the RoPE position of a node is prefix length + depth.

Everything is fp64. The committed prefix keys are already rotated (they were
written at their own positions earlier); the tree's new q and k are rotated here
at position prefix_len + depth. RoPE is the rotate-half form (the page imports
apply_rope without showing it; rotate-half is this oracle's reading).
"""
from __future__ import annotations

import numpy as np

from .tree import position_ids, tree_mask


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta ** (-2 i / D) for i < D/2, fp64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def apply_rope(x, pos, theta: float) -> np.ndarray:
    """Rotate-half RoPE of x [T, ..., D] at integer positions pos [T], fp64.

    out[:D/2] = x1 cos - x2 sin, out[D/2:] = x2 cos + x1 sin, angle = pos * inv_freq.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq(d, theta)[None, :]
    shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (d // 2,)
    cos = np.cos(ang).reshape(shape)
    sin = np.sin(ang).reshape(shape)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def masked_attention(q, keys, values, mask, scale: float) -> np.ndarray:
    """Softmax(q keys^T * scale, masked) values for one head, fp64.

    q [T, D], keys/values [N, D], mask [T, N] bool (True = visible).
    """
    s = (np.asarray(q, np.float64) @ np.asarray(keys, np.float64).T) * scale
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ np.asarray(values, np.float64)


def tree_verify_attention(q, k_new, v_new, k_prefix, v_prefix, parents, theta: float,
                          scale: float):
    """Tree-masked attention of one request.

    q [T, Hq, D], k_new/v_new [T, Hkv, D], k_prefix/v_prefix [Hkv, P, D].
    Returns (out [T, Hq, D], k_rot [T, Hkv, D], v_new [T, Hkv, D]); the last two are
    the keys/values the tree leaves in the cache at slots P .. P+T-1.
    """
    t, hq, _ = q.shape
    hkv = k_new.shape[1]
    p_len = k_prefix.shape[1]
    pos = position_ids(parents, p_len)
    q_rot = apply_rope(q, pos, theta)
    k_rot = apply_rope(k_new, pos, theta)
    full_mask = np.concatenate([np.ones((t, p_len), dtype=bool), tree_mask(parents)], axis=1)
    group = hq // hkv
    out = np.zeros((t, hq, q.shape[2]), dtype=np.float64)
    for kv in range(hkv):
        keys = np.concatenate([np.asarray(k_prefix[kv], np.float64), k_rot[:, kv]], axis=0)
        vals = np.concatenate([np.asarray(v_prefix[kv], np.float64),
                               np.asarray(v_new[:, kv], np.float64)], axis=0)
        for h in range(kv * group, (kv + 1) * group):
            out[:, h] = masked_attention(q_rot[:, h], keys, vals, full_mask, scale)
    return out, k_rot, np.asarray(v_new, np.float64)

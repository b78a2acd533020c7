"""ctypes binding of libtsv.so (the C ABI declared in include/tsv.h).

Argument marshalling only: every function takes torch tensors that already live on the
GPU, checks dtype/shape/contiguity, and forwards raw pointers, sizes and the current
CUDA stream to the library. All computation happens in the library's CUDA kernels.
There is no fallback: if libtsv.so is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtsv.so")

TSV_OK, TSV_ERR_INVALID_ARG, TSV_ERR_UNSUPPORTED, TSV_ERR_WORKSPACE, TSV_ERR_CUDA = range(5)
REQ_CODES = {0: "ok", 1: "bad_root", 2: "bad_parent", 3: "too_deep", 4: "bad_size",
             5: "capacity", 6: "bad_block", 7: "bad_links", 8: "timeout"}
DTYPE_F32, DTYPE_BF16 = 0, 1
KV_CONTIGUOUS, KV_PAGED = 0, 1
KV_BLOCK = 64
MAX_NODES = 256
MAX_TOPK = 16

_c_i32p = ctypes.POINTER(ctypes.c_int32)


class KVCacheDesc(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("layout", ctypes.c_int),
        ("capacity", ctypes.c_int64), ("block_table", ctypes.c_void_p),
        ("max_blocks", ctypes.c_int), ("num_blocks", ctypes.c_int),
        ("num_layers", ctypes.c_int), ("layer_stride", ctypes.c_int64),
    ]


class AttnShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("max_nodes", ctypes.c_int),
                ("num_q_heads", ctypes.c_int), ("max_prefix", ctypes.c_int)]


class TsvError(RuntimeError):
    pass


_lib = None

_SIGNATURES = {
    "tsv_version": (ctypes.c_char_p, []),
    "tsv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tsv_last_cuda_error": (ctypes.c_int, []),
    "tsv_tree_build_meta": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 +
                            [ctypes.c_void_p] * 7 + [ctypes.c_void_p]),
    "tsv_draft_grow_mask": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 +
                            [ctypes.c_void_p] * 2),
    "tsv_draft_topk_expand_workspace_size": (ctypes.c_size_t, [ctypes.c_int] * 4),
    "tsv_draft_topk_expand_launches": (ctypes.c_int, [ctypes.c_int] * 4),
    "tsv_draft_topk_expand": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int] + [ctypes.c_void_p] * 7 +
                              [ctypes.c_size_t, ctypes.c_void_p]),
    "tsv_draft_topk_expand_product": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_int] +
                                      [ctypes.c_void_p] * 7 + [ctypes.c_size_t, ctypes.c_void_p]),
    "tsv_draft_to_target": (ctypes.c_int, [ctypes.c_void_p] * 2 + [ctypes.c_int] * 2 +
                            [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 2),
    "tsv_draft_fixed_level": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int64] + [ctypes.c_int] * 5 +
                              [ctypes.c_void_p] * 3),
    "tsv_draft_select_final": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 +
                               [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 4),
    "tsv_draft_select_tree": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 +
                              [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 4 +
                              [ctypes.c_int] + [ctypes.c_void_p] * 8),
    "tsv_tree_verify_attn_workspace_size": (ctypes.c_size_t, [ctypes.c_void_p] * 2),
    "tsv_tree_verify_attn_launches": (ctypes.c_int, [ctypes.c_void_p] * 2),
    "tsv_tree_verify_attn": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_float] * 2 +
                             [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                              ctypes.c_void_p, ctypes.c_void_p]),
    "tsv_accept_and_compact": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 3 +
                               [ctypes.c_void_p] * 8),
    "tsv_lm_head_argmax_workspace_size": (ctypes.c_size_t, [ctypes.c_int] * 2),
    "tsv_lm_head_argmax": (ctypes.c_int, [ctypes.c_void_p] * 2 + [ctypes.c_int] * 3 +
                           [ctypes.c_void_p] * 3 + [ctypes.c_size_t, ctypes.c_void_p]),
    "tsv_tree_sample_accept_workspace_size": (ctypes.c_size_t, [ctypes.c_int] * 2),
    "tsv_tree_sample_accept": (ctypes.c_int, [ctypes.c_void_p] * 2 + [ctypes.c_int] +
                               [ctypes.c_void_p] * 12 + [ctypes.c_int] * 3 +
                               [ctypes.c_void_p] * 8 + [ctypes.c_size_t, ctypes.c_void_p]),
    "tsv_target_probs": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 5 +
                         [ctypes.c_int] * 2 + [ctypes.c_void_p] * 2 +
                         [ctypes.c_size_t, ctypes.c_void_p]),
    "tsv_tree_verify_attn_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 9 +
                                     [ctypes.c_float] * 2 + [ctypes.c_void_p] * 3),
}
NOALLOC_SCRATCH_BYTES = 32 << 20


def lib():
    """Load libtsv.so (once). Raises if it is missing: there is no fallback path."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise TsvError(f"{LIB_PATH} not found; build it with "
                           "`python -m tree_speculative_decoding_verify_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def exported_symbols():
    return list(_SIGNATURES)


def _check(status: int, what: str):
    if status != TSV_OK:
        msg = lib().tsv_status_string(status).decode()
        if status == TSV_ERR_CUDA:
            msg += f" (cudaError {lib().tsv_last_cuda_error()})"
        raise TsvError(f"{what}: {msg}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t: torch.Tensor, dtype, name: str, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _dtype_code(dt) -> int:
    if dt == torch.bfloat16:
        return DTYPE_BF16
    if dt == torch.float32:
        return DTYPE_F32
    raise TypeError(f"unsupported dtype {dt}")


# ------------------------------------------------------------------------------------
class KVCache:
    """A KV cache as the library sees it (tensors stay owned by the caller).

    contiguous: k, v of shape [num_layers, B, Hkv, capacity, D] or [B, Hkv, capacity, D]
    paged:      k, v of shape [num_layers, num_blocks, Hkv, 64, D] or [num_blocks, Hkv, 64, D]
                plus block_table int32 [B, max_blocks]
    """

    def __init__(self, k: torch.Tensor, v: torch.Tensor, block_table: torch.Tensor = None):
        if k.shape != v.shape or k.dtype != v.dtype:
            raise ValueError("k and v must have the same shape and dtype")
        _need(k, k.dtype, "k")
        _need(v, v.dtype, "v")
        self.k, self.v, self.block_table = k, v, block_table
        layered = k.dim() == 5
        if k.dim() not in (4, 5):
            raise ValueError("k must be 4-D or 5-D")
        self.num_layers = k.shape[0] if layered else 1
        inner = k.shape[1:] if layered else k.shape
        self.paged = block_table is not None
        if self.paged:
            _need(block_table, torch.int32, "block_table")
            if inner[2] != KV_BLOCK:
                raise ValueError("paged blocks must hold 64 tokens")
        self.num_kv_heads = inner[1]
        self.head_dim = inner[3]
        self.dtype = k.dtype
        self.desc = KVCacheDesc(
            k.data_ptr(), v.data_ptr(), _dtype_code(k.dtype), inner[1], inner[3],
            KV_PAGED if self.paged else KV_CONTIGUOUS,
            0 if self.paged else inner[2],
            block_table.data_ptr() if self.paged else None,
            block_table.shape[1] if self.paged else 0,
            inner[0] if self.paged else 0,
            self.num_layers,
            k[0].numel() if layered else 0)

    def layer(self, i: int) -> "KVCache":
        if self.k.dim() != 5:
            return self
        return KVCache(self.k[i], self.v[i], self.block_table)


# ------------------------------------------------------------------------------------
def tree_build_meta(parents, num_nodes, prefix_len, max_depth, mask, position_ids,
                    retrieve_indices, num_leaves, next_token, next_sibling, err=None):
    b, t = parents.shape
    w = (t + 31) // 32
    _need(parents, torch.int32, "parents")
    _need(num_nodes, torch.int32, "num_nodes", (b,))
    _need(prefix_len, torch.int32, "prefix_len", (b,))
    _need(mask, torch.int32, "mask", (b, t, w))
    _need(position_ids, torch.int32, "position_ids", (b, t))
    _need(retrieve_indices, torch.int32, "retrieve_indices", (b, t, max_depth + 1))
    _need(num_leaves, torch.int32, "num_leaves", (b,))
    _need(next_token, torch.int32, "next_token", (b, t))
    _need(next_sibling, torch.int32, "next_sibling", (b, t))
    if err is not None:
        _need(err, torch.int32, "err", (b,))
    _check(lib().tsv_tree_build_meta(_ptr(parents), _ptr(num_nodes), _ptr(prefix_len), b, t,
                                     max_depth, _ptr(mask), _ptr(position_ids),
                                     _ptr(retrieve_indices), _ptr(num_leaves), _ptr(next_token),
                                     _ptr(next_sibling), _ptr(err), _stream()),
           "tsv_tree_build_meta")


def draft_grow_mask(mask, position_ids, new_parents, prefix_len, first_new, err=None):
    """Grow the drafter's mask [B, T, W] (int32 view of the uint32 words) and positions
    [B, T] by one level: new_parents [B, K] int32 (parents of nodes first_new ..
    first_new + K - 1)."""
    b, t = position_ids.shape
    k = new_parents.shape[1]
    _need(mask, torch.int32, "mask", (b, t, (t + 31) // 32))
    _need(position_ids, torch.int32, "position_ids", (b, t))
    _need(new_parents, torch.int32, "new_parents", (b, k))
    _need(prefix_len, torch.int32, "prefix_len", (b,))
    if err is not None:
        _need(err, torch.int32, "err", (b,))
    _check(lib().tsv_draft_grow_mask(_ptr(mask), _ptr(position_ids), _ptr(new_parents),
                                     _ptr(prefix_len), b, first_new, k, t, _ptr(err), _stream()),
           "tsv_draft_grow_mask")


def draft_topk_expand_workspace_size(batch, rows, vocab, top_k) -> int:
    return int(lib().tsv_draft_topk_expand_workspace_size(batch, rows, vocab, top_k))


def draft_topk_expand_launches(batch, rows, vocab, top_k) -> int:
    """Kernels one expansion level of this shape launches (16-byte aligned rows)."""
    return int(lib().tsv_draft_topk_expand_launches(batch, rows, vocab, top_k))


def draft_topk_expand(logits, top_k, level, front_score_in, front_store_in, store_token,
                      store_score, store_parent, front_token_out, front_score_out,
                      front_store_out, workspace, product: bool = False):
    """logits: fp32 [B, rows, V] (last dim may be strided: row stride = logits.stride(1)).
    product: probability-product scores (tsv_draft_topk_expand_product)."""
    if logits.dtype != torch.float32 or not logits.is_cuda or logits.dim() != 3:
        raise TypeError("logits must be a CUDA fp32 tensor [B, rows, V]")
    b, rows, v = logits.shape
    # the stride of a size-1 dimension is meaningless; take the row stride from the
    # first dimension that has more than one entry
    rs = logits.stride(1) if rows > 1 else (logits.stride(0) if b > 1 else v)
    if (v > 1 and logits.stride(2) != 1) or rs < v or (b > 1 and logits.stride(0) != rows * rs):
        raise ValueError("logits rows must be evenly strided with unit element stride")
    cap = store_token.shape[1]
    for name, t, dt in (("store_token", store_token, torch.int32),
                        ("store_score", store_score, torch.float32),
                        ("store_parent", store_parent, torch.int32)):
        _need(t, dt, name, (b, cap))
    for name, t, dt in (("front_token_out", front_token_out, torch.int32),
                        ("front_score_out", front_score_out, torch.float32),
                        ("front_store_out", front_store_out, torch.int32)):
        _need(t, dt, name, (b, top_k))
    if level > 1:
        _need(front_score_in, torch.float32, "front_score_in", (b, rows))
        _need(front_store_in, torch.int32, "front_store_in", (b, rows))
    _need(workspace, torch.uint8, "workspace")
    fn = lib().tsv_draft_topk_expand_product if product else lib().tsv_draft_topk_expand
    _check(fn(
        _ptr(logits), b, rows, rs, v, top_k, level,
        _ptr(front_score_in if level > 1 else None), _ptr(front_store_in if level > 1 else None),
        cap, _ptr(store_token), _ptr(store_score), _ptr(store_parent), _ptr(front_token_out),
        _ptr(front_score_out), _ptr(front_store_out), _ptr(workspace), workspace.numel(),
        _stream()), "tsv_draft_topk_expand")


def draft_to_target(tokens, num_nodes, d2t, err=None):
    """tokens [B, max_nodes] int32 in place: nodes 1 .. num_nodes-1 through the d2t table
    (int32 [draft_vocab])."""
    b, t = tokens.shape
    _need(tokens, torch.int32, "tokens")
    _need(num_nodes, torch.int32, "num_nodes", (b,))
    _need(d2t, torch.int32, "d2t")
    if err is not None:
        _need(err, torch.int32, "err", (b,))
    _check(lib().tsv_draft_to_target(_ptr(tokens), _ptr(num_nodes), b, t, _ptr(d2t), d2t.numel(),
                                     _ptr(err), _stream()), "tsv_draft_to_target")


def draft_fixed_level(logits, width, first_node, first_parent, tokens, parents):
    """One fixed-branching level: logits fp32 [B, frontier, V] (rows evenly strided);
    writes nodes first_node .. first_node + frontier*width - 1 of tokens / parents."""
    if logits.dtype != torch.float32 or not logits.is_cuda or logits.dim() != 3:
        raise TypeError("logits must be a CUDA fp32 tensor [B, frontier, V]")
    b, f, v = logits.shape
    rs = logits.stride(1) if f > 1 else (logits.stride(0) if b > 1 else v)
    if (v > 1 and logits.stride(2) != 1) or rs < v or (b > 1 and logits.stride(0) != f * rs):
        raise ValueError("logits rows must be evenly strided with unit element stride")
    t = tokens.shape[1]
    _need(tokens, torch.int32, "tokens", (b, t))
    _need(parents, torch.int32, "parents", (b, t))
    _check(lib().tsv_draft_fixed_level(_ptr(logits), b, f, rs, v, width, first_node, first_parent,
                                       t, _ptr(tokens), _ptr(parents), _stream()),
           "tsv_draft_fixed_level")


def draft_select_final(store_token, store_score, store_parent, num_candidates, total_tokens,
                       root_token, tokens, parents, num_nodes=None):
    b, cap = store_token.shape
    _need(store_token, torch.int32, "store_token")
    _need(store_score, torch.float32, "store_score", (b, cap))
    _need(store_parent, torch.int32, "store_parent", (b, cap))
    _need(root_token, torch.int32, "root_token", (b,))
    t = tokens.shape[1]
    _need(tokens, torch.int32, "tokens", (b, t))
    _need(parents, torch.int32, "parents", (b, t))
    if num_nodes is not None:
        _need(num_nodes, torch.int32, "num_nodes", (b,))
    _check(lib().tsv_draft_select_final(_ptr(store_token), _ptr(store_score), _ptr(store_parent),
                                        b, num_candidates, cap, total_tokens, _ptr(root_token), t,
                                        _ptr(tokens), _ptr(parents), _ptr(num_nodes), _stream()),
           "tsv_draft_select_final")


def draft_select_tree(store_token, store_score, store_parent, num_candidates, total_tokens,
                      root_token, tokens, parents, num_nodes, prefix_len, max_depth, mask,
                      position_ids, retrieve_indices, num_leaves, next_token, next_sibling,
                      err=None):
    """draft_select_final and tree_build_meta of the selected trees in one launch."""
    b, cap = store_token.shape
    _need(store_token, torch.int32, "store_token")
    _need(store_score, torch.float32, "store_score", (b, cap))
    _need(store_parent, torch.int32, "store_parent", (b, cap))
    _need(root_token, torch.int32, "root_token", (b,))
    t = tokens.shape[1]
    w = (t + 31) // 32
    _need(tokens, torch.int32, "tokens", (b, t))
    _need(parents, torch.int32, "parents", (b, t))
    if num_nodes is not None:
        _need(num_nodes, torch.int32, "num_nodes", (b,))
    _need(prefix_len, torch.int32, "prefix_len", (b,))
    _need(mask, torch.int32, "mask", (b, t, w))
    _need(position_ids, torch.int32, "position_ids", (b, t))
    _need(retrieve_indices, torch.int32, "retrieve_indices", (b, t, max_depth + 1))
    _need(num_leaves, torch.int32, "num_leaves", (b,))
    _need(next_token, torch.int32, "next_token", (b, t))
    _need(next_sibling, torch.int32, "next_sibling", (b, t))
    if err is not None:
        _need(err, torch.int32, "err", (b,))
    _check(lib().tsv_draft_select_tree(_ptr(store_token), _ptr(store_score), _ptr(store_parent),
                                       b, num_candidates, cap, total_tokens, _ptr(root_token), t,
                                       _ptr(tokens), _ptr(parents), _ptr(num_nodes),
                                       _ptr(prefix_len), max_depth, _ptr(mask),
                                       _ptr(position_ids), _ptr(retrieve_indices),
                                       _ptr(num_leaves), _ptr(next_token), _ptr(next_sibling),
                                       _ptr(err), _stream()),
           "tsv_draft_select_tree")


def _attn_shape(q: torch.Tensor, max_prefix: int) -> AttnShape:
    b, t, hq, _ = q.shape
    return AttnShape(b, t, hq, max_prefix)


def tree_verify_attn_workspace_size(q_shape, cache: KVCache, max_prefix: int) -> int:
    b, t, hq, _ = q_shape
    s = AttnShape(b, t, hq, max_prefix)
    return int(lib().tsv_tree_verify_attn_workspace_size(ctypes.byref(s), ctypes.byref(cache.desc)))


def tree_verify_attn_launches(q_shape, cache: KVCache, max_prefix: int) -> int:
    """Kernels one tree_verify_attn call of this shape launches (0: unsupported)."""
    b, t, hq, _ = q_shape
    s = AttnShape(b, t, hq, max_prefix)
    return int(lib().tsv_tree_verify_attn_launches(ctypes.byref(s), ctypes.byref(cache.desc)))


def tree_verify_attn(q, k_new, v_new, cache: KVCache, prefix_len, num_nodes, position_ids, mask,
                     rope_theta, softmax_scale, out, workspace, max_prefix, err=None):
    b, t, hq, d = q.shape
    hkv = cache.num_kv_heads
    _need(q, cache.dtype, "q")
    _need(k_new, cache.dtype, "k_new", (b, t, hkv, d))
    _need(v_new, cache.dtype, "v_new", (b, t, hkv, d))
    _need(out, cache.dtype, "out", (b, t, hq, d))
    _need(prefix_len, torch.int32, "prefix_len", (b,))
    _need(num_nodes, torch.int32, "num_nodes", (b,))
    _need(position_ids, torch.int32, "position_ids", (b, t))
    _need(mask, torch.int32, "mask", (b, t, (t + 31) // 32))
    _need(workspace, torch.uint8, "workspace")
    if err is not None:
        _need(err, torch.int32, "err", (b,))
    s = _attn_shape(q, max_prefix)
    _check(lib().tsv_tree_verify_attn(ctypes.byref(s), _ptr(q), _ptr(k_new), _ptr(v_new),
                                      ctypes.byref(cache.desc), _ptr(prefix_len), _ptr(num_nodes),
                                      _ptr(position_ids), _ptr(mask), float(rope_theta),
                                      float(softmax_scale), _ptr(out), _ptr(workspace),
                                      workspace.numel(), _ptr(err), _stream()),
           "tsv_tree_verify_attn")


def tree_verify_attn_noalloc(q, k_new, v_new, cache: KVCache, prefix_len, num_nodes,
                             position_ids, mask, rope_theta, softmax_scale, out, max_prefix,
                             err=None):
    """tree_verify_attn without a workspace argument, for callers that cannot allocate
    device memory: the library uses a fixed scratch array of NOALLOC_SCRATCH_BYTES per
    device instead (calls on one device share it; see include/tsv.h)."""
    b, t, hq, d = q.shape
    hkv = cache.num_kv_heads
    _need(q, cache.dtype, "q")
    _need(k_new, cache.dtype, "k_new", (b, t, hkv, d))
    _need(v_new, cache.dtype, "v_new", (b, t, hkv, d))
    _need(out, cache.dtype, "out", (b, t, hq, d))
    _need(prefix_len, torch.int32, "prefix_len", (b,))
    _need(num_nodes, torch.int32, "num_nodes", (b,))
    _need(position_ids, torch.int32, "position_ids", (b, t))
    _need(mask, torch.int32, "mask", (b, t, (t + 31) // 32))
    if err is not None:
        _need(err, torch.int32, "err", (b,))
    s = _attn_shape(q, max_prefix)
    _check(lib().tsv_tree_verify_attn_noalloc(ctypes.byref(s), _ptr(q), _ptr(k_new), _ptr(v_new),
                                              ctypes.byref(cache.desc), _ptr(prefix_len),
                                              _ptr(num_nodes), _ptr(position_ids), _ptr(mask),
                                              float(rope_theta), float(softmax_scale), _ptr(out),
                                              _ptr(err), _stream()),
           "tsv_tree_verify_attn_noalloc")


def lm_head_argmax_workspace_size(rows: int, vocab: int) -> int:
    return int(lib().tsv_lm_head_argmax_workspace_size(rows, vocab))


def lm_head_argmax(hidden, weight, argmax, workspace, max_logit=None):
    """argmax[m] = the lowest v maximising hidden[m] . weight[v] (bf16 in, fp32 logits).
    hidden [rows, H] and weight [V, H] bf16; argmax [rows] int32; max_logit [rows] fp32
    or None; workspace uint8 of lm_head_argmax_workspace_size(rows, V) bytes."""
    rows, h = hidden.shape
    v = weight.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight", (v, h))
    _need(argmax, torch.int32, "argmax", (rows,))
    if max_logit is not None:
        _need(max_logit, torch.float32, "max_logit", (rows,))
    _need(workspace, torch.uint8, "workspace")
    _check(lib().tsv_lm_head_argmax(_ptr(hidden), _ptr(weight), rows, h, v, _ptr(argmax),
                                    _ptr(max_logit), _ptr(workspace), workspace.numel(),
                                    _stream()),
           "tsv_lm_head_argmax")


def tree_sample_accept_workspace_size(batch: int, max_nodes: int) -> int:
    return int(lib().tsv_tree_sample_accept_workspace_size(batch, max_nodes))


def _sampling_params(b, temperature, top_k, top_p, min_p):
    _need(temperature, torch.float32, "temperature", (b,))
    _need(top_k, torch.int32, "top_k", (b,))
    _need(top_p, torch.float32, "top_p", (b,))
    _need(min_p, torch.float32, "min_p", (b,))


def tree_sample_accept(target_logits, temperature, top_k, top_p, min_p, u_node, u_final,
                       tokens, next_token, next_sibling, num_nodes, prefix_len, max_depth,
                       cache: Optional[KVCache], accept_path, accept_len, bonus_token, slot_map,
                       new_prefix_len, workspace, err=None, tree_valid=None, draft_probs=None):
    """Non-greedy acceptance (include/tsv.h): target_logits [B, T, V] fp32; per-request
    temperature, top_p, min_p fp32 and top_k int32 [B]; u_node [B, T] and u_final [B]
    uniforms in [0, 1); draft_probs [B, T, V] fp32 or None (target-only)."""
    b, t, v = target_logits.shape
    _need(target_logits, torch.float32, "target_logits")
    if draft_probs is not None:
        _need(draft_probs, torch.float32, "draft_probs", (b, t, v))
    _sampling_params(b, temperature, top_k, top_p, min_p)
    _need(u_node, torch.float32, "u_node", (b, t))
    _need(u_final, torch.float32, "u_final", (b,))
    for name, x in (("tokens", tokens), ("next_token", next_token),
                    ("next_sibling", next_sibling)):
        _need(x, torch.int32, name, (b, t))
    _need(num_nodes, torch.int32, "num_nodes", (b,))
    _need(prefix_len, torch.int32, "prefix_len", (b,))
    _need(accept_path, torch.int32, "accept_path", (b, max_depth + 1))
    _need(accept_len, torch.int32, "accept_len", (b,))
    _need(bonus_token, torch.int32, "bonus_token", (b,))
    _need(slot_map, torch.int32, "slot_map", (b, max_depth + 1, 2))
    _need(new_prefix_len, torch.int32, "new_prefix_len", (b,))
    _need(workspace, torch.uint8, "workspace")
    if err is not None:
        _need(err, torch.int32, "err", (b,))
    if tree_valid is not None:
        _need(tree_valid, torch.int32, "tree_valid", (b,))
    desc = ctypes.byref(cache.desc) if cache is not None else None
    _check(lib().tsv_tree_sample_accept(
        _ptr(target_logits), _ptr(draft_probs), v, _ptr(temperature), _ptr(top_k), _ptr(top_p),
        _ptr(min_p), _ptr(u_node), _ptr(u_final), _ptr(tokens), _ptr(next_token),
        _ptr(next_sibling), _ptr(num_nodes), _ptr(prefix_len), _ptr(tree_valid), b, t,
        max_depth, desc, _ptr(accept_path), _ptr(accept_len), _ptr(bonus_token), _ptr(slot_map),
        _ptr(new_prefix_len), _ptr(err), _ptr(workspace), workspace.numel(), _stream()),
        "tsv_tree_sample_accept")


def target_probs(target_logits, temperature, top_k, top_p, min_p, num_nodes, probs, workspace):
    """The filtered target probabilities [B, T, V] of tree_sample_accept (rows of nodes
    at or past num_nodes are left as they were)."""
    b, t, v = target_logits.shape
    _need(target_logits, torch.float32, "target_logits")
    _need(probs, torch.float32, "probs", (b, t, v))
    _sampling_params(b, temperature, top_k, top_p, min_p)
    _need(num_nodes, torch.int32, "num_nodes", (b,))
    _need(workspace, torch.uint8, "workspace")
    _check(lib().tsv_target_probs(_ptr(target_logits), v, _ptr(temperature), _ptr(top_k),
                                  _ptr(top_p), _ptr(min_p), _ptr(num_nodes), b, t, _ptr(probs),
                                  _ptr(workspace), workspace.numel(), _stream()),
           "tsv_target_probs")


def accept_and_compact(tokens, next_token, next_sibling, target_argmax, num_nodes, prefix_len,
                       max_depth, cache: Optional[KVCache], accept_path, accept_len, bonus_token,
                       slot_map, new_prefix_len, err=None, tree_valid=None):
    b, t = tokens.shape
    for name, x in (("tokens", tokens), ("next_token", next_token),
                    ("next_sibling", next_sibling), ("target_argmax", target_argmax)):
        _need(x, torch.int32, name, (b, t))
    _need(num_nodes, torch.int32, "num_nodes", (b,))
    _need(prefix_len, torch.int32, "prefix_len", (b,))
    _need(accept_path, torch.int32, "accept_path", (b, max_depth + 1))
    _need(accept_len, torch.int32, "accept_len", (b,))
    _need(bonus_token, torch.int32, "bonus_token", (b,))
    _need(slot_map, torch.int32, "slot_map", (b, max_depth + 1, 2))
    _need(new_prefix_len, torch.int32, "new_prefix_len", (b,))
    if err is not None:
        _need(err, torch.int32, "err", (b,))
    if tree_valid is not None:
        _need(tree_valid, torch.int32, "tree_valid", (b,))
    desc = ctypes.byref(cache.desc) if cache is not None else None
    _check(lib().tsv_accept_and_compact(_ptr(tokens), _ptr(next_token), _ptr(next_sibling),
                                        _ptr(target_argmax), _ptr(num_nodes), _ptr(prefix_len),
                                        _ptr(tree_valid), b,
                                        t, max_depth, desc, _ptr(accept_path), _ptr(accept_len),
                                        _ptr(bonus_token), _ptr(slot_map), _ptr(new_prefix_len),
                                        _ptr(err), _stream()),
           "tsv_accept_and_compact")

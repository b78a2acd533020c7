"""GB300-native tree speculative-decoding verification (EAGLE-2/3 dynamic trees).

The compute lives in libtsv.so (hand-written CUDA for sm_103a, C ABI in include/tsv.h);
this package is its Python binding plus a small driver that chains the calls of one
hot-path step over preallocated device buffers.
"""
from ._lib import (  # noqa: F401
    KV_BLOCK, MAX_NODES, MAX_TOPK, REQ_CODES, KVCache, TsvError, accept_and_compact,
    draft_fixed_level, draft_grow_mask, draft_select_final, draft_select_tree, draft_to_target,
    draft_topk_expand, draft_topk_expand_launches, draft_topk_expand_workspace_size, exported_symbols,
    lib, lm_head_argmax, lm_head_argmax_workspace_size, target_probs, tree_build_meta,
    tree_sample_accept, tree_sample_accept_workspace_size, tree_verify_attn,
    tree_verify_attn_launches, tree_verify_attn_noalloc, tree_verify_attn_workspace_size,
)
from .pipeline import HotPath, TreeShape  # noqa: F401

"""One whole pass of the hot path for one request, oracle side (test infrastructure
only): expansion -> final selection -> tree metadata -> tree-masked attention ->
greedy acceptance -> KV compaction. Used to check composed results and to time the
oracle as the CPU baseline."""
from __future__ import annotations

import numpy as np

from . import accept, attention, draft, tree


def hot_path_step(level_logits, top_k: int, total_tokens: int, root_token: int,
                  q, k_new, v_new, k_prefix, v_prefix, target, theta: float, scale: float,
                  retrieve_cols: int):
    """q [T,Hq,D], k_new/v_new [T,Hkv,D], k_prefix/v_prefix [Hkv,P,D]; target is an
    int array [T] or a callable (tokens, parents) -> array."""
    exp = draft.topk_generate(level_logits, top_k)
    tokens, parents = draft.select_final(exp.store_token, exp.store_score, exp.store_parent,
                                         total_tokens, root_token)
    p_len = k_prefix.shape[1]
    mask_words = tree.pack_mask(tree.tree_mask(parents))
    pos = tree.position_ids(parents, p_len)
    retrieve = tree.retrieve_indices(parents, retrieve_cols)
    nxt, sib = tree.next_links(parents)
    out, k_rot, v_tree = attention.tree_verify_attention(q, k_new, v_new, k_prefix, v_prefix,
                                                         parents, theta, scale)
    tgt = target(tokens, parents) if callable(target) else np.asarray(target)
    path, bonus = accept.greedy_walk(tokens, parents, tgt)
    k_all = np.concatenate([np.asarray(k_prefix, np.float64), k_rot.transpose(1, 0, 2)], axis=1)
    v_all = np.concatenate([np.asarray(v_prefix, np.float64), v_tree.transpose(1, 0, 2)], axis=1)
    k_c = accept.compact(k_all, p_len, path)
    v_c = accept.compact(v_all, p_len, path)
    return {
        "tokens": tokens, "parents": parents, "mask": mask_words, "pos": pos,
        "retrieve": retrieve, "next_token": nxt, "next_sibling": sib, "out": out,
        "path": path, "bonus": bonus, "k_cache": k_c, "v_cache": v_c,
        "new_len": p_len + len(path),
    }

"""Seeded cases for the GPU parity tests: inputs from `workloads`, expected values from
`oracle` only (nothing here reads a CUDA result)."""
from __future__ import annotations

import functools
import math

import numpy as np
import torch

import workloads as W
from oracle import draft, tree

BF16_ATOL_MAX = 2e-2     # attention, bf16 inputs: max-abs vs the fp64 oracle
BF16_ATOL_MEAN = 2e-3    # attention, bf16 inputs: mean-abs vs the fp64 oracle
F32_ATOL_MAX = 1e-4      # attention, fp32 inputs (CUDA-core fp32 path) vs fp64
SCORE_RTOL = 1e-5        # fp32 cumulative scores vs the oracle


def dev():
    return torch.device("cuda", 0)


def as_bf16_f64(x: np.ndarray) -> np.ndarray:
    """The values a bf16 tensor holds, as fp64 (what the oracle is given)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).bfloat16().double().numpy()


def to_dev(x: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype).to(dev())


def i32(x) -> torch.Tensor:
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).to(dev())


@functools.lru_cache(maxsize=None)
def level_logits(w: W.Workload, b: int):
    return [W.draft_logits(w, b, lvl) for lvl in range(1, w.depth + 2)]


@functools.lru_cache(maxsize=None)
def oracle_tree(w: W.Workload, b: int):
    """(tokens, parents, expansion) of request b from the oracle's expansion."""
    if w.fixed_parents is not None:
        parents = np.array(w.fixed_parents, dtype=np.int32)
        return W.fixed_tree_tokens(w, b, parents), parents, None
    exp = draft.topk_generate(level_logits(w, b), w.top_k)
    root = int(W.root_tokens(w)[b])
    tokens, parents = draft.select_final(exp.store_token, exp.store_score, exp.store_parent,
                                         w.total_tokens, root)
    return tokens, parents, exp


def random_tree(rng, n: int, max_depth: int):
    """Parent-first random tree of n nodes whose depth stays within max_depth."""
    parents, depth = [-1], [0]
    for i in range(1, n):
        while True:
            p = int(rng.integers(0, i))
            if depth[p] < max_depth:
                break
        parents.append(p)
        depth.append(depth[p] + 1)
    return np.array(parents, dtype=np.int32)


def pad2(rows, width, fill=-1):
    out = np.full((len(rows), width), fill, dtype=np.int32)
    for i, r in enumerate(rows):
        out[i, :len(r)] = r
    return out


def max_depth_of(parents_list):
    return max(max(tree.depths(list(p))) for p in parents_list)


def scale_of(w: W.Workload):
    return 1.0 / math.sqrt(w.head_dim)

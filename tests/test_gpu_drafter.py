"""The drafter's mask grown level by level (tsv_draft_grow_mask) vs the oracle's block
construction, and the drafter's tree attention as tsv_tree_verify_attn over that mask
(bit-exact mask and positions; attention within the bf16 tolerances)."""
import numpy as np
import pytest
import torch

from oracle import tree
from tests import gpu_cases as gc
from tests.test_gpu_attn import Case, make_cache, oracle_one

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def grow(b, k, levels, t_max, prefix, seed):
    """Random K-per-level growth (each new node's parent in the previous level) on the
    GPU; checks every level against the oracle and returns the parents and the device
    mask / positions."""
    import tree_speculative_decoding_verify_gb300 as T
    rng = np.random.default_rng(seed)
    d = gc.dev()
    w = (t_max + 31) // 32
    mask = torch.full((b, t_max, w), -1, dtype=torch.int32, device=d)  # garbage rows
    pos = torch.full((b, t_max), -5, dtype=torch.int32, device=d)
    parents = [[-1] for _ in range(b)]
    o_mask = [np.ones((1, 1), bool) for _ in range(b)]
    o_pos = [np.array([prefix[i]]) for i in range(b)]
    frontier = [[0] for _ in range(b)]
    err = torch.full((b,), 7, dtype=torch.int32, device=d)
    for _ in range(levels):
        n0 = len(parents[0])
        newp = np.array([[frontier[i][int(rng.integers(0, len(frontier[i])))] for _ in range(k)]
                         for i in range(b)], np.int32)
        T.draft_grow_mask(mask, pos, gc.i32(newp), gc.i32(prefix), n0, err)
        torch.cuda.synchronize()
        gm = mask.cpu().numpy().view(np.uint32)
        gp = pos.cpu().numpy()
        for i in range(b):
            o_mask[i], o_pos[i] = tree.grow_level_mask(o_mask[i], o_pos[i], list(newp[i]))
            parents[i] += list(newp[i])
            n = len(parents[i])
            assert (gm[i, :n] == tree.pack_mask(o_mask[i], w)).all()
            assert gp[i, :n].tolist() == o_pos[i].tolist()
            frontier[i] = list(range(n0, n0 + k))
        assert err.cpu().numpy().tolist() == [0] * b
    return parents, mask, pos


def test_grown_mask_matches_block_construction():
    grow(3, 4, 6, 40, [5, 64, 300], seed=1)


def test_bad_parent_is_reported():
    import tree_speculative_decoding_verify_gb300 as T
    d = gc.dev()
    mask = torch.zeros((2, 8, 1), dtype=torch.int32, device=d)
    pos = torch.zeros((2, 8), dtype=torch.int32, device=d)
    err = torch.zeros(2, dtype=torch.int32, device=d)
    T.draft_grow_mask(mask, pos, gc.i32([[0, 0], [0, 0]]), gc.i32([3, 3]), 1, err)
    T.draft_grow_mask(mask, pos, gc.i32([[1, 2], [1, 7]]), gc.i32([3, 3]), 3, err)
    torch.cuda.synchronize()
    assert err.cpu().numpy().tolist() == [0, 2]
    assert pos.cpu().numpy()[1, 4] == -1 and pos.cpu().numpy()[0, 4] == 5


def test_drafter_attention_over_the_grown_mask():
    """The attention of the last level's nodes, with tsv_tree_verify_attn reading the grown
    mask, equals the oracle's tree attention of the grown tree."""
    import tree_speculative_decoding_verify_gb300 as T
    b, k, levels = 2, 4, 5
    t_max = 1 + k * levels
    prefix = [700, 129]
    parents, mask, pos = grow(b, k, levels, t_max, prefix, seed=3)
    c = Case(parents, prefix, 8, 2, 128, torch.bfloat16, seed=4)
    cache, _ = make_cache(c)
    d = gc.dev()
    out = torch.zeros((b, c.t, c.hq, c.d), dtype=torch.bfloat16, device=d)
    ws = torch.empty(T.tree_verify_attn_workspace_size((b, c.t, c.hq, c.d), cache, c.max_prefix),
                     dtype=torch.uint8, device=d)
    T.tree_verify_attn(gc.to_dev(c.q, c.dtype), gc.to_dev(c.k_new, c.dtype),
                       gc.to_dev(c.v_new, c.dtype), cache, gc.i32(c.prefix), gc.i32(c.tn), pos, mask,
                       c.theta, c.scale, out, ws, c.max_prefix)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    g = c.hq // c.hkv
    last = slice(t_max - k, t_max)
    for i in range(b):
        res = oracle_one(c, i)
        for kv, (o, _, _) in res.items():
            diff = np.abs(got[i, last, kv * g:(kv + 1) * g] - o[last])
            assert diff.max() <= gc.BF16_ATOL_MAX and diff.mean() <= gc.BF16_ATOL_MEAN

"""Expansion variants vs the oracle: probability-product scores, the d2t id map and
fixed-branching levels (bit-exact ids and parents; product scores within 1e-5 relative)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import draft
from tests import gpu_cases as gc
from tests.test_gpu_topk import run_levels

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("v,k,depth", [(1000, 4, 3), (32000, 10, 6), (4001, 16, 2)])
def test_product_scores_match_oracle(v, k, depth):
    rng = np.random.default_rng(v + k)
    reqs = [[rng.normal(0, 2, (1 if l == 0 else k, v)).astype(np.float32)
             for l in range(depth + 1)] for _ in range(3)]
    st, ss, sp, hist = run_levels(reqs, k, product=True)
    for b, levels in enumerate(reqs):
        exp = draft.topk_generate(levels, k, product=True)
        c = exp.store_token.size
        np.testing.assert_array_equal(st[b, :c], exp.store_token)
        np.testing.assert_array_equal(sp[b, :c], exp.store_parent)
        np.testing.assert_allclose(ss[b, :c], exp.store_score, rtol=gc.SCORE_RTOL, atol=0)
        # the selections: exact wherever the log-domain margins are clear of fp32 noise
        if draft.margins(draft.topk_generate(levels, k), k) > 1e-4:
            for li, lv in enumerate(exp.levels):
                off = draft.level_store_offset(li + 1, k)
                assert hist[li][2][b].tolist() == [off + f for f in lv.selected], li


def test_product_tree_through_the_step_shape():
    """The dynamic tree from product scores equals the oracle's (tokens, parents)."""
    import tree_speculative_decoding_verify_gb300 as T
    w = W.WORKLOADS["llama8b"]
    d = gc.dev()
    levels = [W.draft_logits(w, 0, lvl) for lvl in range(1, w.depth + 2)]
    exp = draft.topk_generate(levels, w.top_k, product=True)
    root = int(W.root_tokens(w)[0])
    tokens, parents = draft.select_final(exp.store_token, exp.store_score, exp.store_parent,
                                         w.total_tokens, root)
    kc = torch.zeros(1, w.num_kv_heads, 2176, w.head_dim, dtype=torch.bfloat16, device=d)
    shape = T.TreeShape(1, w.num_q_heads, w.num_kv_heads, w.head_dim, 2048, vocab=w.vocab,
                        top_k=w.top_k, depth=w.depth, total_tokens=w.total_tokens,
                        score_product=True)
    hp = T.HotPath(shape, T.KVCache(kc, torch.zeros_like(kc)))
    hp.expand([torch.from_numpy(x[None]).to(d) for x in levels], gc.i32([root]))
    torch.cuda.synchronize()
    assert hp.tokens.cpu().numpy()[0].tolist() == tokens.tolist()
    assert hp.parents.cpu().numpy()[0].tolist() == parents.tolist()


def test_draft_to_target_map():
    import tree_speculative_decoding_verify_gb300 as T
    rng = np.random.default_rng(3)
    b, t, dv = 5, 40, 3000
    d2t = rng.permutation(128256)[:dv].astype(np.int32)
    toks = rng.integers(0, dv, size=(b, t)).astype(np.int32)
    toks[2, 7] = dv + 5      # outside the table
    toks[3, 1] = -2
    nn = np.array([40, 1, 30, 12, 0], np.int32)
    tt = gc.i32(toks)
    err = torch.full((b,), 7, dtype=torch.int32, device=gc.dev())
    T.draft_to_target(tt, gc.i32(nn), gc.i32(d2t), err)
    got = tt.cpu().numpy()
    for i in range(b):
        want = draft.map_draft_to_target(toks[i], int(nn[i]), d2t)
        assert got[i].tolist() == want.tolist(), i
    assert err.cpu().numpy().tolist() == [0, 0, 9, 9, 0]


@pytest.mark.parametrize("v", [1001, 32000])
def test_fixed_branching_levels(v):
    import tree_speculative_decoding_verify_gb300 as T
    rng = np.random.default_rng(v)
    branching = [3, 2, 2]
    b = 4
    rows, frontier = [], 1
    for wdt in branching:
        x = rng.normal(0, 2, (b, frontier, v)).astype(np.float32)
        x[:, :, 5] = x[:, :, 9] = x.max(axis=2) + 1.0   # an exact tie at the top of every row
        rows.append(x)
        frontier *= wdt
    n = 1 + 3 + 6 + 12
    d = gc.dev()
    kc = torch.zeros(b, 1, 64, 64, dtype=torch.bfloat16, device=d)
    shape = T.TreeShape(b, 1, 1, 64, 16, fixed_nodes=n, fixed_max_depth=len(branching))
    hp = T.HotPath(shape, T.KVCache(kc, torch.zeros_like(kc)))
    roots = np.arange(b, dtype=np.int32) + 100
    hp.expand_fixed([torch.from_numpy(x).to(d) for x in rows], gc.i32(roots), branching)
    torch.cuda.synchronize()
    for i in range(b):
        tokens, parents = draft.fixed_tree([x[i] for x in rows], branching, int(roots[i]))
        assert hp.tokens.cpu().numpy()[i].tolist() == tokens.tolist()
        assert hp.parents.cpu().numpy()[i].tolist() == parents.tolist()
    assert (hp.num_nodes.cpu().numpy() == n).all()

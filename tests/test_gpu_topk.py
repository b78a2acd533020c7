"""tsv_draft_topk_expand / tsv_draft_select_final vs the oracle, through the C ABI.
Token ids, parents and store indices are bit-exact; fp32 scores within 1e-5 relative."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import draft
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def run_levels(levels_per_req, k, store_cap=None, stride_pad=0, product=False):
    """Run every level on the GPU; levels_per_req[b][l] is [rows, V] fp32 numpy."""
    import tree_speculative_decoding_verify_gb300 as T
    b = len(levels_per_req)
    nlev = len(levels_per_req[0])
    v = levels_per_req[0][0].shape[1]
    cap = store_cap or draft.num_candidates(k, nlev - 1)
    d = gc.dev()
    st = torch.full((b, cap), -7, dtype=torch.int32, device=d)
    ss = torch.full((b, cap), -7.0, dtype=torch.float32, device=d)
    sp = torch.full((b, cap), -7, dtype=torch.int32, device=d)
    fronts = [(torch.zeros(b, k, dtype=torch.int32, device=d),
               torch.zeros(b, k, dtype=torch.float32, device=d),
               torch.zeros(b, k, dtype=torch.int32, device=d)) for _ in range(2)]
    ws_n = max(T.draft_topk_expand_workspace_size(b, r, v, k) for r in (1, k))
    ws = torch.zeros(ws_n, dtype=torch.uint8, device=d)  # zeroed once, reused by every level
    history = []
    cur = None
    for li in range(nlev):
        rows = levels_per_req[0][li].shape[0]
        host = np.zeros((b, rows, v + stride_pad), dtype=np.float32)
        for bi in range(b):
            host[bi, :, :v] = levels_per_req[bi][li]
        lg = torch.from_numpy(host).to(d)[:, :, :v]
        nxt = fronts[li % 2]
        T.draft_topk_expand(lg, k, li + 1, None if cur is None else cur[1],
                            None if cur is None else cur[2], st, ss, sp, *nxt, ws,
                            product=product)
        torch.cuda.synchronize()
        history.append(tuple(t.cpu().numpy().copy() for t in nxt))
        # the per-request counters at the start of the workspace are back at zero
        assert not ws[:4 * b].view(torch.int32).any().item()
        cur = nxt
    return st.cpu().numpy(), ss.cpu().numpy(), sp.cpu().numpy(), history


def compare(levels_per_req, k, **kw):
    st, ss, sp, hist = run_levels(levels_per_req, k, **kw)
    for b, levels in enumerate(levels_per_req):
        exp = draft.topk_generate(levels, k)
        c = exp.store_token.size
        np.testing.assert_array_equal(st[b, :c], exp.store_token)
        np.testing.assert_array_equal(sp[b, :c], exp.store_parent)
        np.testing.assert_allclose(ss[b, :c], exp.store_score, rtol=gc.SCORE_RTOL, atol=0)
        for li, lv in enumerate(exp.levels):
            off = draft.level_store_offset(li + 1, k)
            ft, fs, fi = hist[li]
            assert fi[b].tolist() == [off + f for f in lv.selected], f"level {li + 1}"
            assert ft[b].tolist() == [int(lv.tokens[f]) for f in lv.selected]
    return st, ss, sp


@pytest.mark.parametrize("b", [3, 80])
@pytest.mark.parametrize("v", [64, 1000, 4001, 32000])
def test_levels_small_and_ragged_vocab(v, b):
    """3 requests take the row-per-CTA cluster kernel at every level; 80 requests of 4
    rows (320 rows, more than two waves of the GPU's SMs) take the per-unit kernel from
    level 2 on."""
    rng = np.random.default_rng(v + b)
    k, depth = 4, 3
    reqs = [[(rng.standard_normal((1 if l == 0 else k, v)) * 2).astype(np.float32)
             for l in range(depth + 1)] for _ in range(b)]
    compare(reqs, k)


@pytest.mark.parametrize("v,k,b,pad,product", [
    (32768, 16, 4, 0, False),    # the longest row and the largest cluster (16 rows)
    (32767, 16, 3, 1, False),    # stride 32768 but ragged: 128-bit loads, a partial group
    (30001, 10, 6, 0, False),    # unaligned rows: scalar loads
    (30001, 10, 6, 3, True),     # aligned ragged rows, product scores
    (32000, 8, 4, 0, False),     # clusters of 8 (the long-prefix workload's shape)
    (32000, 10, 16, 0, False),   # 160 rows: the clusters run in two waves (serving's shape)
    (20, 16, 2, 0, False),       # fewer threads with entries than k: every entry survives
])
def test_row_clusters(v, k, b, pad, product):
    """Small batches: one CTA per frontier row holds the whole row in registers and the
    request's rows form a thread-block cluster whose rank-0 CTA runs the joint top-K over
    distributed shared memory. Every level is compared with the oracle."""
    rng = np.random.default_rng(v + 7 * k + b + pad)
    reqs = [[(rng.standard_normal((1 if l == 0 else k, v)) * 2).astype(np.float32)
             for l in range(3)] for _ in range(b)]
    if product:
        st, ss, sp, hist = run_levels(reqs, k, stride_pad=pad, product=True)
        for bi, levels in enumerate(reqs):
            exp = draft.topk_generate(levels, k, product=True)
            c = exp.store_token.size
            np.testing.assert_array_equal(st[bi, :c], exp.store_token)
            np.testing.assert_array_equal(sp[bi, :c], exp.store_parent)
            np.testing.assert_allclose(ss[bi, :c], exp.store_score, rtol=gc.SCORE_RTOL, atol=0)
    else:
        compare(reqs, k, stride_pad=pad)


@pytest.mark.parametrize("v", [32768, 5000])
def test_row_clusters_constant_rows(v):
    """Rows whose entries are all equal: every warp's and thread's best entry ties in value,
    so the bounds are decided by index alone and hundreds of thread maxima reach the first
    bound; the top k must be the k lowest ids of every row."""
    k, b = 16, 2
    reqs = [[np.full((1 if l == 0 else k, v), 0.25 * (l + 1), dtype=np.float32)
             for l in range(2)] for _ in range(b)]
    st, ss, sp = compare(reqs, k)
    assert st[0, :k].tolist() == list(range(k))


def test_strided_rows_and_max_topk():
    rng = np.random.default_rng(5)
    k, v = 16, 3000
    reqs = [[(rng.standard_normal((1 if l == 0 else k, v)) * 2).astype(np.float32)
             for l in range(3)] for _ in range(2)]
    compare(reqs, k, stride_pad=12)
    compare(reqs, k, stride_pad=3)        # unaligned row stride -> scalar loads


def test_exact_ties_go_to_lower_ids():
    rng = np.random.default_rng(9)
    k, v = 5, 777
    reqs = []
    for _ in range(2):
        l1 = rng.integers(-3, 3, size=(1, v)).astype(np.float32)
        l2 = np.tile(rng.integers(-3, 3, size=(1, v)).astype(np.float32), (k, 1))  # equal rows
        reqs.append([l1, l2])
    st, ss, sp = compare(reqs, k)
    assert st.shape[1] == k + k * k


def test_llama8b_expansion_and_final_selection():
    import tree_speculative_decoding_verify_gb300 as T
    w = W.WORKLOADS["llama8b"]
    levels = gc.level_logits(w, 0)
    st, ss, sp = compare([levels], w.top_k)
    tokens, parents, exp = gc.oracle_tree(w, 0)
    assert draft.margins(exp, w.total_tokens) > 0
    d = gc.dev()
    tok = torch.zeros(1, w.num_nodes + 3, dtype=torch.int32, device=d)
    par = torch.zeros_like(tok)
    nn = torch.zeros(1, dtype=torch.int32, device=d)
    T.draft_select_final(gc.i32(st), torch.from_numpy(ss).to(d), gc.i32(sp), w.num_candidates,
                         w.total_tokens, gc.i32(W.root_tokens(w)), tok, par, nn)
    torch.cuda.synchronize()
    assert tok.cpu().numpy()[0, :w.num_nodes].tolist() == tokens.tolist()
    assert par.cpu().numpy()[0, :w.num_nodes].tolist() == parents.tolist()
    assert tok.cpu().numpy()[0, w.num_nodes:].tolist() == [-1] * 3
    assert nn.item() == w.num_nodes


@pytest.mark.parametrize("name", ["long70b", "serving"])
def test_workload_trees(name):
    w = W.WORKLOADS[name]
    nreq = 4 if name == "serving" else 1
    compare([gc.level_logits(w, b) for b in range(nreq)], w.top_k)


def test_sweep_level_640_rows_of_128256():
    """One level of the batch-64 sweep: logits [64 x 10, 128256]; rows checked on a
    sample of requests against the oracle's per-row top-k and log-probabilities."""
    import tree_speculative_decoding_verify_gb300 as T
    w = W.WORKLOADS["sweep"]
    k = w.top_k
    host = np.stack([W.draft_logits(w, b, 2) for b in range(w.batch)])   # [64, 10, V]
    d = gc.dev()
    lg = torch.from_numpy(host).to(d)
    cap = draft.num_candidates(k, w.depth)
    st = torch.zeros(w.batch, cap, dtype=torch.int32, device=d)
    ss = torch.zeros(w.batch, cap, dtype=torch.float32, device=d)
    sp = torch.zeros(w.batch, cap, dtype=torch.int32, device=d)
    fin_s = torch.zeros(w.batch, k, dtype=torch.float32, device=d)
    fin_i = (torch.arange(k, dtype=torch.int32, device=d) + 100).repeat(w.batch, 1)
    outs = [torch.zeros(w.batch, k, dtype=torch.int32, device=d),
            torch.zeros(w.batch, k, dtype=torch.float32, device=d),
            torch.zeros(w.batch, k, dtype=torch.int32, device=d)]
    ws = torch.zeros(T.draft_topk_expand_workspace_size(w.batch, k, w.vocab, k),
                     dtype=torch.uint8, device=d)
    T.draft_topk_expand(lg, k, 2, fin_s, fin_i, st, ss, sp, *outs, ws)
    torch.cuda.synchronize()
    st, ss, sp = st.cpu().numpy(), ss.cpu().numpy(), sp.cpu().numpy()
    for b in (0, 17, 63):
        lv = draft.expand_level(host[b], k, np.zeros(k, np.float32), np.arange(k) + 100)
        np.testing.assert_array_equal(st[b, k:k + k * k], lv.tokens)
        np.testing.assert_array_equal(sp[b, k:k + k * k], lv.parent_store)
        np.testing.assert_allclose(ss[b, k:k + k * k], lv.cu, rtol=gc.SCORE_RTOL)
        assert outs[2].cpu().numpy()[b].tolist() == [k + f for f in lv.selected]


@pytest.mark.parametrize("pad", [1, 0])
def test_whole_row_units_ragged_vocab(pad):
    """640 frontier rows put whole rows in one unit each (one CTA streams 40003 entries):
    the row's last three entries fall outside the 16-byte groups; stride 40004 keeps rows
    16-byte aligned (vector loads), stride 40003 does not (scalar loads)."""
    rng = np.random.default_rng(40003 + pad)
    k, v, b = 10, 40003, 64
    reqs = [[(rng.standard_normal((1 if l == 0 else k, v)) * 2).astype(np.float32)
             for l in range(2)] for _ in range(b)]
    compare(reqs, k, stride_pad=pad)


@pytest.mark.parametrize("v", [2048, 2049, 4001, 4096])
def test_two_step_units_in_registers(v):
    """320 frontier rows of at most 4096 entries give one unit per row of one or two
    128-bit steps: every entry stays in registers and the unit's top k comes from the
    CTA-wide bound and survivor ranking (2048: exactly one step; 2049: a second step with
    a single entry; 4001: a ragged second step; 4096: two full steps)."""
    rng = np.random.default_rng(v)
    k, b = 10, 32
    reqs = [[(rng.standard_normal((1 if l == 0 else k, v)) * 2).astype(np.float32)
             for l in range(2)] for _ in range(b)]
    compare(reqs, k)


@pytest.mark.parametrize("v,k,b,pad,product", [
    (40000, 10, 64, 0, False),   # 640 rows: shares of 4.2 rows, rows split between CTAs
    (40000, 10, 64, 4, True),    # padded (still 16-byte aligned) rows, product scores
    (32000, 16, 24, 0, False),   # the largest top_k: 384 rows, shares just over a row
    (40000, 10, 64, 1, False),   # unaligned stride: the per-unit kernel, same layout
])
def test_large_batch_shares(v, k, b, pad, product):
    """Large batches take the persistent kernel (one CTA per SM over an equal share of all
    rows' entries, so a row may be split between two CTAs); every level is compared with
    the oracle: tokens, parents and frontier exactly, scores within 1e-5."""
    rng = np.random.default_rng(v + k + pad)
    reqs = [[(rng.standard_normal((1 if l == 0 else k, v)) * 2).astype(np.float32)
             for l in range(2)] for _ in range(b)]
    if product:
        st, ss, sp, hist = run_levels(reqs, k, stride_pad=pad, product=True)
        for bi, levels in enumerate(reqs):
            exp = draft.topk_generate(levels, k, product=True)
            c = exp.store_token.size
            np.testing.assert_array_equal(st[bi, :c], exp.store_token)
            np.testing.assert_array_equal(sp[bi, :c], exp.store_parent)
            np.testing.assert_allclose(ss[bi, :c], exp.store_score, rtol=gc.SCORE_RTOL, atol=0)
    else:
        compare(reqs, k, stride_pad=pad)


def _select_expected(score, parent, total):
    """Kept store indices (the oracle's ordering: score, then lower index) and the tree
    they form; a kept candidate whose parent was not kept hangs from the root (node 0)."""
    best = sorted(draft.topk_by_score(score, total))
    node_of = {c: i + 1 for i, c in enumerate(best)}
    par = [-1] + [node_of.get(int(parent[c]), 0) if parent[c] >= 0 else 0 for c in best]
    return best, par


@pytest.mark.parametrize("case", ["spread", "coarse_ties", "all_equal", "narrow_bin",
                                  "keep_all", "keep_one", "signed_zeros"])
def test_select_final_thresholds(case):
    """The final selection on synthetic stores: spread scores (one histogram pass and a
    few candidates ranked in the threshold bin), scores on a coarse grid (ties inside the
    bin), all-equal scores and a bin of about 600 candidates (the radix-select fallback),
    every candidate kept, a single one kept, and -0 / +0 ties."""
    import tree_speculative_decoding_verify_gb300 as T
    rng = np.random.default_rng(sum(map(ord, case)))
    C, total = 4096, 60
    if case == "spread":
        score = (rng.standard_normal(C) * 4 - 10).astype(np.float32)
    elif case == "coarse_ties":
        C = 610
        score = np.round(rng.standard_normal(C) * 3 - 8).astype(np.float32)
    elif case == "all_equal":
        score = np.full(C, -3.5, dtype=np.float32)
    elif case == "narrow_bin":
        C = 3000
        score = (-8.0 - rng.random(C) * 0.9).astype(np.float32)  # one 12-bit bin
        total = 100
    elif case == "keep_all":
        C = 250  # total_tokens + 1 nodes, at most 256
        score = (rng.standard_normal(C) - 5).astype(np.float32)
        total = C
    elif case == "keep_one":
        score = (rng.standard_normal(C) - 5).astype(np.float32)
        total = 1
    else:
        C = 200
        score = np.where(rng.random(C) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
        score[::7] = -1.0
        total = 50
    parent = np.array([-1 if c < 10 else int(rng.integers(0, c)) for c in range(C)], np.int32)
    token = (np.arange(C) + 1000).astype(np.int32)
    d = gc.dev()
    nodes = total + 1
    tok = torch.zeros(1, nodes + 2, dtype=torch.int32, device=d)
    par = torch.zeros_like(tok)
    nn = torch.zeros(1, dtype=torch.int32, device=d)
    T.draft_select_final(gc.i32(token[None]), torch.from_numpy(score[None]).to(d),
                         gc.i32(parent[None]), C, total, gc.i32(np.array([7], np.int32)),
                         tok, par, nn)
    torch.cuda.synchronize()
    best, exp_par = _select_expected(score, parent, total)
    got_tok = tok.cpu().numpy()[0]
    assert got_tok[0] == 7 and nn.item() == nodes
    assert (got_tok[1:nodes] - 1000).tolist() == best
    assert par.cpu().numpy()[0, :nodes].tolist() == exp_par
    assert got_tok[nodes:].tolist() == [-1, -1]


def test_select_tree_matches_the_two_calls():
    """tsv_draft_select_tree (selection and metadata in one launch) against
    tsv_draft_select_final followed by tsv_tree_build_meta on the same stores: every
    output identical, on three expanded requests with different prefix lengths."""
    import tree_speculative_decoding_verify_gb300 as T
    w = W.WORKLOADS["llama8b"]
    k, depth, total = w.top_k, w.depth, w.total_tokens
    reqs = [gc.level_logits(w, 0)]
    rng = np.random.default_rng(31)
    for _ in range(2):
        reqs.append([(rng.standard_normal((1 if l == 0 else k, w.vocab)) * 2).astype(np.float32)
                     for l in range(depth + 1)])
    st, ss, sp, _ = run_levels(reqs, k)
    d = gc.dev()
    b, t, cols = len(reqs), w.num_nodes + 3, depth + 2
    words = (t + 31) // 32
    st, ss, sp = gc.i32(st), torch.from_numpy(ss).to(d), gc.i32(sp)
    root = gc.i32(np.array([5, 6, 7], np.int32))
    prefix = gc.i32(np.array([2048, 17, 0], np.int32))

    def outs():
        z = lambda *shape: torch.full(shape, -9, dtype=torch.int32, device=d)
        return dict(tok=z(b, t), par=z(b, t), nn=z(b), mask=z(b, t, words), pos=z(b, t),
                    ret=z(b, t, cols), nl=z(b), nt=z(b, t), ns=z(b, t), err=z(b))

    a, c = outs(), outs()
    T.draft_select_final(st, ss, sp, w.num_candidates, total, root, a["tok"], a["par"], a["nn"])
    T.tree_build_meta(a["par"], a["nn"], prefix, cols - 1, a["mask"], a["pos"], a["ret"],
                      a["nl"], a["nt"], a["ns"], a["err"])
    T.draft_select_tree(st, ss, sp, w.num_candidates, total, root, c["tok"], c["par"], c["nn"],
                        prefix, cols - 1, c["mask"], c["pos"], c["ret"], c["nl"], c["nt"],
                        c["ns"], c["err"])
    torch.cuda.synchronize()
    for name in a:
        assert torch.equal(a[name], c[name]), name
    assert c["err"].cpu().tolist() == [0, 0, 0]
    tokens, parents, _ = gc.oracle_tree(w, 0)
    assert c["tok"].cpu().numpy()[0, :w.num_nodes].tolist() == [5] + tokens.tolist()[1:]


def test_row_clusters_masked_rows():
    """Rows that are -inf except for three tokens (a masked vocabulary): two of every
    row's five candidates are -inf tokens, taken by lower id, and the value bound leaves
    every entry, so the exact bound runs."""
    k = 5
    rng = np.random.default_rng(77 + k)
    v, b = 32000, 3
    reqs = []
    for _ in range(b):
        lv = []
        for l in range(3):
            rows = 1 if l == 0 else k
            x = np.full((rows, v), -np.inf, dtype=np.float32)
            for r in range(rows):
                idx = rng.choice(v, size=3, replace=False)
                x[r, idx] = rng.standard_normal(3).astype(np.float32) * 2
            lv.append(x)
        reqs.append(lv)
    st, ss, sp, _ = run_levels(reqs, k)
    for bi, levels in enumerate(reqs):
        exp = draft.topk_generate(levels, k)
        c = exp.store_token.size
        np.testing.assert_array_equal(st[bi, :c], exp.store_token)
        np.testing.assert_array_equal(sp[bi, :c], exp.store_parent)
        fin = np.isfinite(exp.store_score)
        assert np.array_equal(np.isfinite(ss[bi, :c]), fin)
        np.testing.assert_allclose(ss[bi, :c][fin], exp.store_score[fin], rtol=gc.SCORE_RTOL)


def test_row_clusters_tied_maxima():
    """Every row holds its largest value four times (at random ids) over a spread of
    smaller ones: the ties at the top go to the lower ids."""
    rng = np.random.default_rng(91)
    k, v, b = 6, 30000, 3
    reqs = []
    for _ in range(b):
        lv = []
        for l in range(3):
            rows = 1 if l == 0 else k
            x = (rng.standard_normal((rows, v)) * 2).astype(np.float32)
            for r in range(rows):
                x[r, rng.choice(v, size=4, replace=False)] = np.float32(9.5)
            lv.append(x)
        reqs.append(lv)
    compare(reqs, k)

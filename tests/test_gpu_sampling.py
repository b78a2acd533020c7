"""tsv_target_probs and tsv_tree_sample_accept vs the sampling oracle.

The kernels form masses in fp32 (2^((l - m) log2(e) / T)) and add them with compensated
fp32 sums in a fixed order; the oracle works in fp64. Probabilities must agree within
1e-5 relative (plus 2^-38 absolute for masses far below anything that can decide), and
kept sets must be equal except for tokens the fp64 reading puts within 1e-5 of a top-p or
min-p boundary. For the walk, path and token must be equal on every request whose
decisions all lie further than 1e-5 from flipping (the oracle's trace says how far each
one was); the others (expected to be rare) are counted and bounded.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import accept, sampling, tree
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu

PARAMS = [  # (temperature, top_k, top_p, min_p)
    (1.0, 0, 1.0, 0.0), (0.7, 50, 1.0, 0.0), (1.3, 0, 0.9, 0.0), (1.0, 40, 0.8, 0.05),
    (0.0, 0, 1.0, 0.0), (0.5, 5000, 0.95, 0.01), (1.0, 1, 1.0, 0.0), (2.0, 0, 0.5, 0.0),
    (1.0, 0, 1.0, 0.2), (0.8, 3, 0.3, 0.0), (1.5, 70000, 0.99, 0.0), (1.0, 7, 1.0, 0.9),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def params_t(params):
    d = gc.dev()
    t = torch.tensor([p[0] for p in params], dtype=torch.float32, device=d)
    k = torch.tensor([p[1] for p in params], dtype=torch.int32, device=d)
    pp = torch.tensor([p[2] for p in params], dtype=torch.float32, device=d)
    mp = torch.tensor([p[3] for p in params], dtype=torch.float32, device=d)
    return t, k, pp, mp


def run_probs(logits, params, num_nodes):
    import tree_speculative_decoding_verify_gb300 as T
    b, t, v = logits.shape
    d = gc.dev()
    lt = torch.from_numpy(logits).to(d)
    out = torch.full((b, t, v), -1.0, dtype=torch.float32, device=d)
    ws = torch.empty(T.tree_sample_accept_workspace_size(b, t), dtype=torch.uint8, device=d)
    T.target_probs(lt, *params_t(params), gc.i32(num_nodes), out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def borderline(lg, prm, tol=1e-5):
    """Tokens whose membership the fp64 reading puts within tol of a top-p or min-p
    boundary (either side may keep them)."""
    tau, k, pp, mp = prm
    lg = np.where(np.isnan(lg), -np.inf, lg.astype(np.float64))
    if not tau > 0 or k == 1 or pp <= 0 or not np.isfinite(lg.max()):
        return set()
    e = np.exp((lg - lg.max()) / tau)
    order = np.lexsort((np.arange(len(lg)), -lg))
    if 0 < k < len(lg):
        order = order[:k]
    out = set()
    if pp < 1:
        total = e[order].sum()
        before = np.concatenate([[0.0], np.cumsum(e[order])[:-1]])
        out |= set(order[np.abs(before - pp * total) <= tol * total].tolist())
    if mp > 0:
        out |= set(np.flatnonzero(np.abs(e - min(mp, 1.0)) <= tol).tolist())
    return out


def check_probs(got, logits, params, num_nodes):
    for b, prm in enumerate(params):
        for i in range(num_nodes[b]):
            want = sampling.filter_probs(logits[b, i], *prm)
            g = got[b, i].astype(np.float64)
            diff = np.flatnonzero((g > 0) != (want > 0))
            allowed = borderline(logits[b, i], prm) | set(np.flatnonzero(want < 2.0 ** -38).tolist())
            assert set(diff.tolist()) <= allowed, (b, i, prm, diff[:10])
            both = (g > 0) & (want > 0)
            np.testing.assert_array_less(np.abs(g[both] - want[both]),
                                         1e-5 * want[both] + 2.0 ** -38)


@pytest.mark.parametrize("vocab", [32000, 50001, 128256])
def test_filtered_probabilities(vocab):
    b, t = len(PARAMS), 3
    rng = np.random.default_rng(vocab)
    logits = (rng.standard_normal((b, t, vocab), dtype=np.float32) * 2).astype(np.float32)
    logits[0, 1, 100:140] = logits[0, 1, 99]          # a tie group
    logits[3, 0, ::3] = -np.inf                        # masked entries
    logits[5, 2, :] = np.round(logits[5, 2, :], 1)     # many exact ties
    logits[9, 1, 10] = logits[9, 1].max()              # a tie for the maximum
    logits[7, 2, :] = 1.0  # one tie group of the whole row: top-p 0.5 keeps the lower half
                           # by id, more tokens than the sorted list holds (radix select)
    nn = [t] * b
    nn[2] = 1  # rows of absent nodes are left alone
    got = run_probs(logits, PARAMS, nn)
    check_probs(got, logits, PARAMS, nn)
    assert (got[2, 1:] == -1.0).all()
    kept = np.flatnonzero(got[7, 2] > 0)
    assert kept.tolist() == list(range((vocab + 1) // 2))


def _links(parents, t_max):
    nt, ns = tree.next_links(list(parents))
    a = np.full(t_max, -1, np.int32)
    s = np.full(t_max, -1, np.int32)
    a[:len(parents)], s[:len(parents)] = nt, ns
    return a, s


def make_case(w, nreq, vocab, t_max, params, seed, draft=False, max_depth=None):
    """Random parent-first trees (siblings carry distinct tokens), logits boosted along a
    planted walk, uniforms, and (draft-aware) a draft distribution per node."""
    rng = np.random.default_rng(seed)
    trees = []
    for b in range(nreq):
        n = int(rng.integers(1, t_max + 1))
        parents = [-1] + [int(rng.integers(max(0, i - 4), i)) for i in range(1, n)]
        tokens = [int(rng.integers(0, vocab))]
        for i in range(1, n):
            used = {tokens[j] for j in range(1, i) if parents[j] == parents[i]}
            x = int(rng.integers(0, vocab))
            while x in used:
                x = int(rng.integers(0, vocab))
            tokens.append(x)
        trees.append((np.array(tokens, np.int32), np.array(parents, np.int32)))
    md = max_depth or max(max(tree.depths(list(p))) for _, p in trees)
    logits = np.stack([W.target_logits(w, b, tk, pr, vocab, t_max) for b, (tk, pr) in
                       enumerate(trees)])
    u = np.stack([W.uniforms(w, b, t_max) for b in range(nreq)])
    q = None
    if draft:
        dl = np.stack([W.target_logits(w, b, tk, pr, vocab, t_max, stream="d_logits")
                       for b, (tk, pr) in enumerate(trees)]).astype(np.float64)
        q = np.exp(dl - dl.max(axis=2, keepdims=True))
        q = (q / q.sum(axis=2, keepdims=True)).astype(np.float32)
    prm = [params[b % len(params)] for b in range(nreq)]
    return trees, md, logits, u, q, prm


def run_walk(trees, md, logits, u, q, prm, t_max, cache=None, prefix=None, valid=None,
             nn=None):
    import tree_speculative_decoding_verify_gb300 as T
    d = gc.dev()
    b = len(trees)
    tok = np.full((b, t_max), -1, np.int32)
    nxt = np.full((b, t_max), -1, np.int32)
    sib = np.full((b, t_max), -1, np.int32)
    for i, (tk, pr) in enumerate(trees):
        tok[i, :len(tk)] = tk
        nxt[i], sib[i] = _links(pr, t_max)
    out = dict(accept_path=torch.full((b, md + 1), 9, dtype=torch.int32, device=d),
               accept_len=torch.zeros(b, dtype=torch.int32, device=d),
               bonus_token=torch.zeros(b, dtype=torch.int32, device=d),
               slot_map=torch.zeros(b, md + 1, 2, dtype=torch.int32, device=d),
               new_prefix_len=torch.zeros(b, dtype=torch.int32, device=d),
               err=torch.full((b,), 9, dtype=torch.int32, device=d))
    ws = torch.empty(T.tree_sample_accept_workspace_size(b, t_max), dtype=torch.uint8, device=d)
    T.tree_sample_accept(
        torch.from_numpy(logits).to(d), *params_t(prm),
        torch.from_numpy(np.ascontiguousarray(u[:, :t_max])).to(d),
        torch.from_numpy(np.ascontiguousarray(u[:, t_max])).to(d),
        gc.i32(tok), gc.i32(nxt), gc.i32(sib),
        gc.i32(nn if nn is not None else [len(tk) for tk, _ in trees]),
        gc.i32(prefix if prefix is not None else [0] * b), md, cache, out["accept_path"],
        out["accept_len"], out["bonus_token"], out["slot_map"], out["new_prefix_len"], ws,
        err=out["err"], tree_valid=None if valid is None else gc.i32(valid),
        draft_probs=None if q is None else torch.from_numpy(q).to(d))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def oracle_walk(trees, logits, u, q, prm, t_max, valid=None):
    """Per request: (path, token, margin of the acceptance tests, final distribution)."""
    res = []
    for b, (tk, pr) in enumerate(trees):
        n = len(tk)
        probs = [sampling.filter_probs(logits[b, i], *prm[b]) for i in range(n)]
        qq = None if q is None else [q[b, i].astype(np.float64) for i in range(n)]
        trace = []
        path, tok = sampling.rejection_walk(list(tk), list(pr), probs, u[b, :t_max],
                                            float(u[b, t_max]), qq,
                                            True if valid is None else bool(valid[b]), trace)
        tests = [abs(x - a) for kind, x, a in trace if kind == "test"]
        final = [(x, p) for kind, x, p in trace if kind == "final"][-1]
        res.append((path, tok, min(tests, default=1.0), final))
    return res


def valid_sample(t, final, tol=1e-6):
    """Token t is what the inverse CDF of the final distribution gives for a u within
    tol of the given one."""
    u, p = final
    c = np.cumsum(p) / p.sum()
    lo = c[t - 1] if t > 0 else 0.0
    return 0 <= t < len(p) and p[t] > 0 and lo - tol <= u <= c[t] + tol


def compare(got, want, tol=1e-5, max_close=0.03):
    """Paths equal wherever every acceptance test is further than tol from flipping;
    tokens equal, or (a near-tie of the inverse CDF) a valid sample of the oracle's final
    distribution."""
    close = other = 0
    for b, (path, tok, margin, final) in enumerate(want):
        n = int(got["accept_len"][b])
        gpath, gtok = got["accept_path"][b, :n].tolist(), int(got["bonus_token"][b])
        if margin < tol:
            close += 1
            continue
        assert gpath == path, (b, gpath, path)
        assert got["err"][b] == 0
        if gtok != tok:
            assert valid_sample(gtok, final), (b, gtok, tok)
            other += 1
    assert close <= max(1, max_close * len(want)), close
    assert other <= max(1, max_close * len(want)), other


@pytest.mark.parametrize("draft", [False, True])
@pytest.mark.parametrize("vocab", [1000, 32001])
def test_walk_matches_oracle(draft, vocab):
    w = W.WORKLOADS["llama8b"]
    t_max = 24
    trees, md, logits, u, q, prm = make_case(w, 48, vocab, t_max, PARAMS, seed=vocab + draft,
                                             draft=draft)
    got = run_walk(trees, md, logits, u, q, prm, t_max)
    want = oracle_walk(trees, logits, u, q, prm, t_max)
    compare(got, want)
    # the walk goes somewhere: some requests accept beyond the root
    assert (got["accept_len"] > 1).sum() >= 5


def test_zero_temperature_is_the_greedy_acceptance():
    """temperature 0 everywhere: the path and bonus of the greedy walk given the target's
    argmax, for any uniforms."""
    w = W.WORKLOADS["llama8b"]
    t_max = 20
    trees, md, logits, u, q, prm = make_case(w, 32, 500, t_max, [(0.0, 0, 1.0, 0.0)], seed=11)
    got = run_walk(trees, md, logits, u, q, prm, t_max)
    for b, (tk, pr) in enumerate(trees):
        n = len(tk)
        target = [int(np.argmax(logits[b, i])) for i in range(n)]
        path, bonus = accept.greedy_walk(list(tk), list(pr), target)
        assert got["accept_path"][b, :got["accept_len"][b]].tolist() == path
        assert got["bonus_token"][b] == bonus


def test_invalid_tree_and_bad_size():
    w = W.WORKLOADS["llama8b"]
    t_max = 8
    trees, md, logits, u, q, prm = make_case(w, 4, 300, t_max, [(1.0, 0, 1.0, 0.0)], seed=5)
    got = run_walk(trees, md, logits, u, q, prm, t_max, valid=[1, 0, 1, 0])
    want = oracle_walk(trees, logits, u, q, prm, t_max, valid=[1, 0, 1, 0])
    compare(got, want, max_close=0.5)
    assert got["accept_len"][1] == 1 and got["accept_len"][3] == 1
    # a request whose node count is out of range: root only, no token, TSV_REQ_BAD_SIZE
    nn = [len(tk) for tk, _ in trees]
    nn[2] = 0
    bad = run_walk(trees, md, logits, u, q, prm, t_max, nn=nn)
    assert bad["err"][2] == 4 and bad["accept_len"][2] == 1 and bad["bonus_token"][2] == -1
    assert bad["accept_path"][2].tolist() == [0] + [-1] * md


def test_llama8b_and_serving_shapes():
    """Every node of one Llama-3-8B-vocabulary tree (61 nodes x 128256) and a batch of 16
    such trees, top-p / top-k / temperature mixes, against the oracle."""
    w = W.WORKLOADS["serving"]
    t_max = 61
    prm_mix = [(1.0, 0, 0.9, 0.0), (0.7, 50, 1.0, 0.0), (1.0, 20, 0.8, 0.05), (0.0, 0, 1.0, 0.0)]
    trees, md, logits, u, q, prm = make_case(w, 16, 128256, t_max, prm_mix, seed=61)
    got = run_walk(trees, md, logits, u, q, prm, t_max)
    want = oracle_walk(trees, logits, u, q, prm, t_max)
    compare(got, want)
    probs = run_probs(logits[:2], prm[:2], [len(trees[0][0]), len(trees[1][0])])
    check_probs(probs, logits[:2], prm[:2], [len(trees[0][0]), len(trees[1][0])])


def test_compaction_follows_the_sampled_path():
    """The cache after the call equals the oracle's compaction along the oracle's
    rejection-walk path (requests whose decisions are all clear of flipping)."""
    import tree_speculative_decoding_verify_gb300 as T
    w = W.WORKLOADS["llama8b"]
    t_max, P = 16, 40
    trees, md, logits, u, q, prm = make_case(w, 6, 400, t_max, [(1.0, 0, 1.0, 0.0)], seed=21)
    d = gc.dev()
    cap = 64 * 2
    kc = torch.randn(6, 2, cap, 64, device=d).to(torch.bfloat16)
    vc = torch.randn(6, 2, cap, 64, device=d).to(torch.bfloat16)
    k0, v0 = kc.float().cpu().numpy(), vc.float().cpu().numpy()
    got = run_walk(trees, md, logits, u, q, prm, t_max, cache=T.KVCache(kc, vc), prefix=[P] * 6)
    want = oracle_walk(trees, logits, u, q, prm, t_max)
    kk, vv = kc.float().cpu().numpy(), vc.float().cpu().numpy()
    checked = 0
    for b, (path, _, margin, _) in enumerate(want):
        n = int(got["accept_len"][b])
        if margin < 1e-5:
            continue
        assert got["accept_path"][b, :n].tolist() == path
        np.testing.assert_array_equal(kk[b], accept.compact(k0[b], P, path))
        np.testing.assert_array_equal(vv[b], accept.compact(v0[b], P, path))
        assert got["new_prefix_len"][b] == P + len(path)
        checked += 1
    assert checked >= 5

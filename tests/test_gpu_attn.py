"""tsv_tree_verify_attn vs the fp64 oracle, through the C ABI.

bf16 inputs: max-abs <= 2e-2 and mean-abs <= 2e-3; fp32 inputs: max-abs <= 1e-4.
The cache afterwards holds the tree's rotated keys (within one bf16 rounding step of
the oracle's fp64 keys) and its values (bit-exact), and zeros up to the next slot that
is a multiple of 16."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention, tree
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


class Case:
    """Host inputs of one attention call (fp32 draws; rounded to dtype on upload)."""

    def __init__(self, parents_list, prefix, hq, hkv, d, dtype, t_max=None, paged=False,
                 seed=0, scale_values=None, theta=1e4, capacity=None, max_prefix=None):
        rng = np.random.default_rng(seed)
        self.b = len(parents_list)
        self.parents = [np.asarray(p, dtype=np.int32) for p in parents_list]
        self.tn = np.array([len(p) for p in self.parents], dtype=np.int32)
        self.t = t_max or int(self.tn.max())
        self.prefix = np.asarray(prefix, dtype=np.int32)
        self.hq, self.hkv, self.d, self.dtype, self.paged, self.theta = hq, hkv, d, dtype, paged, theta
        sv = scale_values if scale_values is not None else (
            1.0 / math.sqrt(d) if dtype == torch.bfloat16 else 1.0)
        f = lambda *s: (rng.standard_normal(s, dtype=np.float32) * np.float32(sv))
        self.q = f(self.b, self.t, hq, d)
        self.k_new = f(self.b, self.t, hkv, d)
        self.v_new = f(self.b, self.t, hkv, d)
        self.k_pre = [f(hkv, int(p), d) for p in self.prefix]
        self.v_pre = [f(hkv, int(p), d) for p in self.prefix]
        self.max_prefix = max_prefix if max_prefix is not None else int(self.prefix.max())
        self.capacity = capacity or int(math.ceil((self.max_prefix + self.t + 16) / 64) * 64)
        self.scale = 1.0 / math.sqrt(d)

    def rounded(self, x):
        return gc.as_bf16_f64(x) if self.dtype == torch.bfloat16 else np.asarray(x, np.float64)


def make_cache(c: Case):
    import tree_speculative_decoding_verify_gb300 as T
    dev = gc.dev()
    if not c.paged:
        # slots past the prefix hold NaN: a kernel that reads a slot it should not
        # turns the output non-finite
        k = torch.full((c.b, c.hkv, c.capacity, c.d), float("nan"), dtype=c.dtype, device=dev)
        v = torch.full_like(k, float("nan"))
        for b in range(c.b):
            p = int(c.prefix[b])
            k[b, :, :p] = gc.to_dev(c.k_pre[b], c.dtype)
            v[b, :, :p] = gc.to_dev(c.v_pre[b], c.dtype)
        return T.KVCache(k, v), None
    per = c.capacity // 64
    pool = c.b * per + 3
    rng = np.random.default_rng(1234)
    table = rng.permutation(pool)[:c.b * per].reshape(c.b, per).astype(np.int32)
    k = torch.full((pool, c.hkv, 64, c.d), float("nan"), dtype=c.dtype, device=dev)
    v = torch.full_like(k, float("nan"))
    for b in range(c.b):
        p = int(c.prefix[b])
        kp = gc.to_dev(c.k_pre[b], c.dtype)
        vp = gc.to_dev(c.v_pre[b], c.dtype)
        for s0 in range(0, p, 64):
            n = min(64, p - s0)
            blk = int(table[b, s0 // 64])
            k[blk, :, :n] = kp[:, s0:s0 + n]
            v[blk, :, :n] = vp[:, s0:s0 + n]
    return T.KVCache(k, v, gc.i32(table)), table


def logical_rows(cache, table, b, kv, slots):
    """Cache rows of request b, kv head kv at the given slots (host copies)."""
    if table is None:
        return cache.k[b, kv, slots].float().cpu().numpy(), cache.v[b, kv, slots].float().cpu().numpy()
    ks, vs = [], []
    for s in slots:
        blk = int(table[b, s // 64])
        ks.append(cache.k[blk, kv, s % 64].float().cpu().numpy())
        vs.append(cache.v[blk, kv, s % 64].float().cpu().numpy())
    return np.stack(ks), np.stack(vs)


def run(c: Case, err=None):
    import tree_speculative_decoding_verify_gb300 as T
    dev = gc.dev()
    cache, table = make_cache(c)
    w = (c.t + 31) // 32
    mask = np.zeros((c.b, c.t, w), dtype=np.uint32)
    pos = np.zeros((c.b, c.t), dtype=np.int32)
    for b, p in enumerate(c.parents):
        n = len(p)
        mask[b, :n] = tree.pack_mask(tree.tree_mask(list(p)), w)
        pos[b, :n] = tree.position_ids(list(p), int(c.prefix[b]))
    out = torch.full((c.b, c.t, c.hq, c.d), 777.0, dtype=c.dtype, device=dev)
    ws = torch.empty(T.tree_verify_attn_workspace_size((c.b, c.t, c.hq, c.d), cache, c.max_prefix),
                     dtype=torch.uint8, device=dev)
    err_t = torch.full((c.b,), 9, dtype=torch.int32, device=dev)
    T.tree_verify_attn(gc.to_dev(c.q, c.dtype), gc.to_dev(c.k_new, c.dtype),
                       gc.to_dev(c.v_new, c.dtype), cache, gc.i32(c.prefix), gc.i32(c.tn),
                       gc.i32(pos), torch.from_numpy(mask.view(np.int32)).to(dev), c.theta,
                       c.scale, out, ws, c.max_prefix, err_t)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), cache, table, err_t.cpu().numpy()


def oracle_one(c: Case, b, kvs=None):
    n = int(c.tn[b])
    kvs = range(c.hkv) if kvs is None else kvs
    g = c.hq // c.hkv
    res = {}
    for kv in kvs:
        sl = slice(kv * g, (kv + 1) * g)
        out, k_rot, v_new = attention.tree_verify_attention(
            c.rounded(c.q[b, :n, sl]), c.rounded(c.k_new[b, :n, kv:kv + 1]),
            c.rounded(c.v_new[b, :n, kv:kv + 1]), c.rounded(c.k_pre[b][kv:kv + 1]),
            c.rounded(c.v_pre[b][kv:kv + 1]), list(c.parents[b]), c.theta, c.scale)
        res[kv] = (out, k_rot[:, 0], v_new[:, 0])
    return res


def check(c: Case, samples=None):
    got, cache, table, err = run(c)
    assert (err == 0).all(), err
    g = c.hq // c.hkv
    pairs = samples or [(b, kv) for b in range(c.b) for kv in range(c.hkv)]
    diffs = []
    for b, kv in pairs:
        n = int(c.tn[b])
        out, k_rot, v_new = oracle_one(c, b, [kv])[kv]
        diffs.append(np.abs(got[b, :n, kv * g:(kv + 1) * g] - out).ravel())
        p = int(c.prefix[b])
        pad_end = ((p + n + 15) // 16) * 16        # zeros up to this slot
        ks, vs = logical_rows(cache, table, b, kv, list(range(p, pad_end)))
        tol = 2.0 ** -7 if c.dtype == torch.bfloat16 else 1e-6
        np.testing.assert_allclose(ks[:n], k_rot, rtol=tol, atol=1e-6)
        np.testing.assert_array_equal(vs[:n], v_new)
        assert (ks[n:] == 0).all() and (vs[n:] == 0).all()
        # rows past the tree are zero
        assert (got[b, n:] == 0).all()
    for b in range(c.b):
        bad = [kv for kv in range(c.hkv) if not np.isfinite(got[b, :, kv * g:(kv + 1) * g]).all()]
        assert not bad, f"non-finite output: request {b}, kv heads {bad}"
    d = np.concatenate(diffs)
    if c.dtype == torch.bfloat16:
        assert d.max() <= gc.BF16_ATOL_MAX, d.max()
        assert d.mean() <= gc.BF16_ATOL_MEAN, d.mean()
    else:
        assert d.max() <= gc.F32_ATOL_MAX, d.max()
    return d


def test_tiny_fp32_page_tree():
    w = W.WORKLOADS["tiny"]
    c = Case([w.fixed_parents], [32], 4, 2, 64, torch.float32)
    check(c)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_batch_edges(dtype, d):
    rng = np.random.default_rng(d)
    trees = [[-1], [-1, 0], gc.random_tree(rng, 33, 6), gc.random_tree(rng, 61, 7),
             gc.random_tree(rng, 5, 3), tree.kary_parents(40, 1)]
    prefix = [0, 1, 127, 128, 129, 300]
    check(Case(trees, prefix, 8, 2, d, dtype, t_max=64, seed=d))


@pytest.mark.parametrize("paged", [False, True])
def test_unaligned_prefixes_never_read_past_the_tree(paged):
    rng = np.random.default_rng(21)
    trees = [gc.random_tree(rng, n, 7) for n in (61, 13, 1, 49, 30, 2)]
    prefix = [1000, 777, 3, 129, 510, 4093]   # P + T at every residue mod 16
    check(Case(trees, prefix, 16, 4, 128, torch.bfloat16, seed=22, paged=paged))


def test_llama8b_contiguous():
    w = W.WORKLOADS["llama8b"]
    _, parents, _ = gc.oracle_tree(w, 0)
    check(Case([parents], [w.max_prefix], w.num_q_heads, w.num_kv_heads, w.head_dim,
               torch.bfloat16, seed=11))


def test_serving_paged():
    w = W.WORKLOADS["serving"]
    prefix = W.prefix_lengths(w)
    trees = [gc.oracle_tree(w, b)[1] for b in range(w.batch)]
    c = Case(trees, prefix, w.num_q_heads, w.num_kv_heads, w.head_dim, torch.bfloat16,
             paged=True, seed=12, max_prefix=w.max_prefix)
    check(c, samples=[(b, kv) for b in range(w.batch) for kv in (0, 5)])


def test_long70b_sampled():
    w = W.WORKLOADS["long70b"]
    _, parents, _ = gc.oracle_tree(w, 0)
    c = Case([parents] * w.batch, [w.max_prefix] * w.batch, w.num_q_heads, w.num_kv_heads,
             w.head_dim, torch.bfloat16, seed=13)
    # eight (request, KV head) pairs: every request twice, every KV head once
    check(c, samples=[(0, 0), (0, 7), (1, 2), (1, 5), (2, 1), (2, 6), (3, 3), (3, 4)])


@pytest.mark.parametrize("total", W.SWEEP_TOTAL_TOKENS)
def test_sweep_sampled(total):
    w = W.WORKLOADS["sweep"]
    rng = np.random.default_rng(total)
    trees = [gc.random_tree(rng, total + 1, w.depth + 1) for _ in range(w.batch)]
    c = Case(trees, [w.max_prefix] * w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
             torch.bfloat16, seed=14)
    # eight (request, KV head) pairs spread over the batch, every KV head once
    check(c, samples=[(9 * i, i) for i in range(8)])


def test_request_that_does_not_fit_is_rejected_on_device():
    trees = [[-1, 0, 0], [-1, 0, 1, 2, 3]]     # 60 + 5 slots (rounded to 80) > 64
    c = Case(trees, [40, 60], 4, 2, 128, torch.bfloat16, capacity=64, max_prefix=60)
    got, cache, _, err = run(c)
    assert err.tolist() == [0, 5]
    assert (got[1] == 0).all() and np.isfinite(got[0]).all()
    # the rejected request's cache is untouched (NaN from setup)
    assert torch.isnan(cache.k[1, :, 60:].float()).all()

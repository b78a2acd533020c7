"""tsv_lm_head_argmax vs the oracle: the target's greedy token at every node.

The kernel forms the logits in fp32 on the tensor cores, the oracle in fp64 from the
same bf16 values. Where a row's best logit leads the runner-up by more than twice the
fp32 accumulation bound the two must name the same token; closer than that, the
kernel's token must still be a valid argmax (its exact logit within the bound of the
best). The reported maximum logit is the exact logit of the returned token within the
bound. Bound per row: hidden_size * 2^-23 * max_v sum_k |h_k w_vk| (the usual
n * unit-roundoff bound of a recursive sum, doubled for the two roundings of a
fused add).
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import lm_head
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def bf16_np(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).bfloat16().float().numpy()


def make_inputs(w, rows, hidden, vocab, key=0):
    """Device bf16 hidden and weight, and the fp32 copies of the same bf16 values."""
    h = bf16_np(W.lm_head_hidden(w, rows, hidden, key))
    wt = torch.empty(vocab, hidden, dtype=torch.bfloat16, device=gc.dev())
    w_host = np.empty((vocab, hidden), np.float32)
    for v0, blk in W.lm_head_weight_blocks(w, vocab, hidden, key):
        t = torch.from_numpy(blk).bfloat16()
        wt[v0:v0 + blk.shape[0]] = t.to(gc.dev())
        w_host[v0:v0 + blk.shape[0]] = t.float().numpy()
    return torch.from_numpy(h).bfloat16().to(gc.dev()), wt, h, w_host


def run(hidden_t, weight_t):
    import tree_speculative_decoding_verify_gb300 as T
    rows, v = hidden_t.shape[0], weight_t.shape[0]
    am = torch.full((rows,), -7, dtype=torch.int32, device=gc.dev())
    ml = torch.full((rows,), float("nan"), dtype=torch.float32, device=gc.dev())
    ws = torch.empty(max(T.lm_head_argmax_workspace_size(rows, v), 256), dtype=torch.uint8,
                     device=gc.dev())
    T.lm_head_argmax(hidden_t, weight_t, am, ws, ml)
    torch.cuda.synchronize()
    return am.cpu().numpy(), ml.cpu().numpy()


def check(h, w_host, am, ml, sample=None):
    """h [rows, H] fp32 (bf16 values); compare the rows in `sample` (all by default)."""
    rows, hdim = h.shape
    sample = np.arange(rows) if sample is None else np.asarray(sample)
    hs = h[sample].astype(np.float64)
    idx, best = lm_head.lm_head_argmax(hs, w_host)
    got = am[sample]
    assert ((got >= 0) & (got < w_host.shape[0])).all(), "index out of range"
    # the bound and the runner-up, per sampled row (fp64 logits, chunked like the oracle)
    absmax = np.zeros(len(sample))
    second = np.full(len(sample), -np.inf)
    for v0 in range(0, w_host.shape[0], 8192):
        blk = w_host[v0:v0 + 8192].astype(np.float64)
        absmax = np.maximum(absmax, (np.abs(hs) @ np.abs(blk).T).max(axis=1))
        lg = hs @ blk.T
        cols = np.arange(v0, v0 + blk.shape[0])
        lg[cols[None, :] == idx[:, None]] = -np.inf
        second = np.maximum(second, lg.max(axis=1))
    tol = hdim * 2.0 ** -23 * absmax
    exact_at_got = np.einsum("rk,rk->r", hs, w_host[got].astype(np.float64))
    clear = best - second > 2 * tol
    assert (got[clear] == idx[clear]).all(), \
        f"rows {sample[clear][got[clear] != idx[clear]].tolist()} differ with a clear gap"
    assert (exact_at_got >= best - tol).all(), "a returned token is not a valid argmax"
    np.testing.assert_array_less(np.abs(ml[sample] - exact_at_got), tol + 1e-30)
    # the bound is a worst case; actual fp32 errors are far smaller, so near-ties that
    # the bound cannot separate still come out equal almost always
    return int((got == idx).sum()), len(sample)


@pytest.mark.parametrize("rows,hidden,vocab", [
    (1, 64, 1), (3, 64, 255), (5, 64, 257), (61, 128, 1000), (128, 192, 4097),
    (129, 64, 513), (300, 256, 30001),
])
def test_small_and_ragged(rows, hidden, vocab):
    w = W.WORKLOADS["tiny"]
    ht, wt, h, w_host = make_inputs(w, rows, hidden, vocab, key=rows * 7 + vocab)
    am, ml = run(ht, wt)
    same, n = check(h, w_host, am, ml)
    assert same >= n - 2


def test_llama8b_every_node():
    """The 61 nodes of one Llama-3-8B-shaped tree against the full 128256-entry head."""
    w = W.WORKLOADS["llama8b"]
    hdim, vocab = W.TARGET_LM_HEAD["llama8b"]
    ht, wt, h, w_host = make_inputs(w, w.batch * w.num_nodes, hdim, vocab)
    am, ml = run(ht, wt)
    same, n = check(h, w_host, am, ml)
    assert same >= n - 2


@pytest.mark.parametrize("name", ["serving", "sweep"])
def test_many_row_tiles_sampled(name):
    """Every node of the batch (8 and 33 row tiles), sampled rows against the oracle."""
    w = W.WORKLOADS[name]
    hdim, vocab = W.TARGET_LM_HEAD[name]
    rows = w.batch * w.num_nodes
    ht, wt, h, w_host = make_inputs(w, rows, hdim, vocab)
    am, ml = run(ht, wt)
    rng = np.random.default_rng(5)
    sample = np.unique(np.concatenate([[0, 127, 128, rows - 1],
                                       rng.choice(rows, 40, replace=False)]))
    same, n = check(h, w_host, am, ml, sample)
    assert same >= n - 2


def test_equal_rows_go_to_the_lowest_index():
    """Identical weight rows in different vocabulary splits tie exactly: the first wins."""
    w = W.WORKLOADS["tiny"]
    rows, hdim, vocab = 40, 128, 40000
    ht, wt, h, w_host = make_inputs(w, rows, hdim, vocab, key=99)
    sign = np.where(W.lm_head_hidden(w, 1, hdim, 98)[0] >= 0, 1.0, -1.0).astype(np.float32)
    h = np.abs(h) * sign[None, :]          # every row aligned with the planted direction
    dup = (37000, 20000, 4100, 4099)       # the winner 4 * sign, planted four times
    for c in dup:
        w_host[c] = 4 * sign
    wt[list(dup)] = torch.from_numpy(np.stack([4 * sign] * len(dup))).bfloat16().to(gc.dev())
    ht = torch.from_numpy(h).bfloat16().to(gc.dev())
    am, ml = run(ht, wt)
    idx, best = lm_head.lm_head_argmax(h.astype(np.float64), w_host)
    assert (idx == min(dup)).all()
    assert (am == min(dup)).all(), am
    np.testing.assert_allclose(ml, best, rtol=1e-5)


def test_all_logits_negative():
    """Negative logits everywhere: the least negative is the answer (ordering of the
    sign-flipped keys)."""
    w = W.WORKLOADS["tiny"]
    rows, hdim, vocab = 9, 64, 3000
    h = np.abs(bf16_np(W.lm_head_hidden(w, rows, hdim, 3))) + 0.25
    w_host = -np.abs(bf16_np(next(W.lm_head_weight_blocks(w, vocab, hdim, 3))[1])) - 0.01
    w_host = bf16_np(w_host)
    h = bf16_np(h)
    am, ml = run(torch.from_numpy(h).bfloat16().to(gc.dev()),
                 torch.from_numpy(w_host).bfloat16().to(gc.dev()))
    assert (ml < 0).all()
    check(h, w_host, am, ml)


def test_zero_rows_and_bad_arguments():
    import tree_speculative_decoding_verify_gb300 as T
    d = gc.dev()
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=d)
    wt = torch.zeros(100, 64, dtype=torch.bfloat16, device=d)
    T.lm_head_argmax(torch.zeros(0, 64, dtype=torch.bfloat16, device=d), wt,
                     torch.zeros(0, dtype=torch.int32, device=d), ws)
    with pytest.raises(T.TsvError):  # hidden size not a multiple of 64
        T.lm_head_argmax(torch.zeros(2, 96, dtype=torch.bfloat16, device=d),
                         torch.zeros(100, 96, dtype=torch.bfloat16, device=d),
                         torch.zeros(2, dtype=torch.int32, device=d), ws)
    with pytest.raises(T.TsvError):  # workspace too small
        T.lm_head_argmax(torch.zeros(200, 64, dtype=torch.bfloat16, device=d), wt,
                         torch.zeros(200, dtype=torch.int32, device=d), ws[:8])

"""tsv_tree_verify_attn_noalloc: the attention call for callers that cannot allocate device
memory (their memory is owned by their own pool, or their loop must not call cudaMalloc,
which can synchronize the device). It runs on a fixed scratch array inside the library
instead of a caller workspace; these tests check that two calls in a row give the same
results as tsv_tree_verify_attn on the same inputs and as the fp64 oracle, and that a
shape needing more scratch than the array holds is refused."""
import math

import numpy as np
import pytest
import torch

from oracle import attention, tree
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def inputs(seed, b=2, hq=32, hkv=8, d=128, p_len=1500, n=61, cap=1664):
    rng = np.random.default_rng(seed)
    dev = gc.dev()
    s = 1 / math.sqrt(d)
    f = lambda *shape: torch.from_numpy(rng.standard_normal(shape, dtype=np.float32) * np.float32(s))
    parents = [gc.random_tree(rng, n, 7) for _ in range(b)]
    w = (n + 31) // 32
    mask = np.zeros((b, n, w), dtype=np.uint32)
    pos = np.zeros((b, n), dtype=np.int32)
    for i, par in enumerate(parents):
        mask[i] = tree.pack_mask(tree.tree_mask(list(par)), w)
        pos[i] = tree.position_ids(list(par), p_len)
    k = f(b, hkv, cap, d).to(torch.bfloat16).to(dev)
    v = f(b, hkv, cap, d).to(torch.bfloat16).to(dev)
    return dict(q=f(b, n, hq, d).to(torch.bfloat16).to(dev),
                k_new=f(b, n, hkv, d).to(torch.bfloat16).to(dev),
                v_new=f(b, n, hkv, d).to(torch.bfloat16).to(dev),
                k=k, v=v, prefix=gc.i32([p_len] * b), nodes=gc.i32([n] * b), pos=gc.i32(pos),
                mask=torch.from_numpy(mask.view(np.int32)).to(dev), p_len=p_len, parents=parents)


def oracle_out(x, b):
    """The fp64 oracle's attention output of request b (from the bf16 values the call got)."""
    f64 = lambda t: t.double().cpu().numpy()
    p_len = x["p_len"]
    out, _, _ = attention.tree_verify_attention(
        f64(x["q"][b]), f64(x["k_new"][b]), f64(x["v_new"][b]), f64(x["k"][b, :, :p_len]),
        f64(x["v"][b, :, :p_len]), list(x["parents"][b]), 1e4, 1 / math.sqrt(x["q"].shape[-1]))
    return out


def run(x, noalloc):
    import tree_speculative_decoding_verify_gb300 as T
    k, v = x["k"].clone(), x["v"].clone()
    cache = T.KVCache(k, v)
    out = torch.full_like(x["q"], 7.0)
    err = torch.full((x["q"].shape[0],), 9, dtype=torch.int32, device=gc.dev())
    args = (x["q"], x["k_new"], x["v_new"], cache, x["prefix"], x["nodes"], x["pos"], x["mask"],
            1e4, 1 / math.sqrt(x["q"].shape[-1]))
    if noalloc:
        T.tree_verify_attn_noalloc(*args, out, x["p_len"], err)
    else:
        ws = torch.empty(T.tree_verify_attn_workspace_size(tuple(x["q"].shape), cache, x["p_len"]),
                         dtype=torch.uint8, device=gc.dev())
        T.tree_verify_attn(*args, out, ws, x["p_len"], err)
    return out, k, v, err


def test_two_calls_in_a_row_match_the_workspace_call():
    first, second = inputs(1), inputs(2, p_len=700, n=33)
    got = [run(first, True), run(second, True)]       # back to back on the shared scratch
    torch.cuda.synchronize()
    for x, (out, k, v, err) in zip((first, second), got):
        ref_out, ref_k, ref_v, ref_err = run(x, False)
        torch.cuda.synchronize()
        assert err.tolist() == [0, 0] and ref_err.tolist() == [0, 0]
        diff = (out.float() - ref_out.float()).abs()
        assert diff.max().item() <= gc.BF16_ATOL_MAX
        assert diff.mean().item() <= gc.BF16_ATOL_MEAN
        assert torch.equal(k, ref_k) and torch.equal(v, ref_v)
        # and directly against the fp64 oracle, every output of every request
        for b in range(x["q"].shape[0]):
            want = oracle_out(x, b)
            d = np.abs(out[b].float().cpu().numpy().astype(np.float64) - want)
            assert d.max() <= gc.BF16_ATOL_MAX and d.mean() <= gc.BF16_ATOL_MEAN, (d.max(), d.mean())


def test_shape_beyond_the_scratch_is_refused():
    import tree_speculative_decoding_verify_gb300 as T
    x = inputs(3, b=2)
    cache = T.KVCache(x["k"], x["v"])
    huge_prefix = 1 << 24          # split partials for this bound exceed the scratch
    need = T.tree_verify_attn_workspace_size(tuple(x["q"].shape), cache, huge_prefix)
    assert need > T._lib.NOALLOC_SCRATCH_BYTES
    out = torch.zeros_like(x["q"])
    with pytest.raises(T.TsvError, match="workspace"):
        T.tree_verify_attn_noalloc(x["q"], x["k_new"], x["v_new"], cache, x["prefix"], x["nodes"],
                                   x["pos"], x["mask"], 1e4, 0.088, out, huge_prefix)

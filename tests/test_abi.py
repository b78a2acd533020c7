"""The C-ABI library builds for sm_103a, loads, exports every symbol include/tsv.h
declares, and rejects bad arguments on the host (these calls return before any CUDA
work, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

from tree_speculative_decoding_verify_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "tsv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tsv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for want in ("tsv_draft_topk_expand", "tsv_draft_select_final", "tsv_tree_build_meta",
                 "tsv_tree_verify_attn", "tsv_accept_and_compact"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(_lib.exported_symbols())


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.tsv_version()
    assert lib.tsv_status_string(0) == b"ok"
    assert lib.tsv_status_string(3).startswith(b"workspace")


def test_host_validation_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: the checks fail first
    # build_meta: max_nodes out of range
    assert lib.tsv_tree_build_meta(p, p, p, 1, 0, 4, p, p, p, p, p, p, None, None) == 1
    assert lib.tsv_tree_build_meta(p, p, p, 1, 257, 4, p, p, p, p, p, p, None, None) == 1
    # topk: top_k too large; rows inconsistent with level; store too small
    assert lib.tsv_draft_topk_expand(p, 1, 1, 100, 100, 17, 1, None, None, 100,
                                     p, p, p, p, p, p, p, 1 << 20, None) == 1
    assert lib.tsv_draft_topk_expand(p, 1, 2, 100, 100, 4, 1, None, None, 100,
                                     p, p, p, p, p, p, p, 1 << 20, None) == 1
    assert lib.tsv_draft_topk_expand(p, 1, 4, 100, 100, 4, 3, p, p, 10,
                                     p, p, p, p, p, p, p, 1 << 20, None) == 1
    # topk: workspace too small
    assert lib.tsv_draft_topk_expand(p, 1, 1, 100, 100, 4, 1, None, None, 100,
                                     p, p, p, p, p, p, p, 8, None) == 3
    # select_final: total_tokens above the candidate count
    assert lib.tsv_draft_select_final(p, p, p, 1, 10, 10, 11, p, 64, p, p, None, None) == 1
    # select_tree: the same check, a depth past TSV_MAX_DEPTH, a missing metadata array;
    # an empty batch is a no-op
    meta = [p] * 6 + [None]
    assert lib.tsv_draft_select_tree(p, p, p, 1, 10, 10, 11, p, 64, p, p, None, p, 8, *meta,
                                     None) == 1
    assert lib.tsv_draft_select_tree(p, p, p, 1, 10, 10, 5, p, 64, p, p, None, p, 99, *meta,
                                     None) == 1
    assert lib.tsv_draft_select_tree(p, p, p, 1, 10, 10, 5, p, 64, p, p, None, p, 8, None,
                                     *meta[1:], None) == 1
    assert lib.tsv_draft_select_tree(None, None, None, 0, 10, 10, 5, None, 64, None, None, None,
                                     None, 8, *([None] * 7), None) == 0
    # attention: unsupported head_dim, GQA mismatch, missing workspace
    k = ctypes.c_void_p(256)
    cache = _lib.KVCacheDesc(k, k, 1, 8, 96, 0, 128, None, 0, 0, 1, 0)
    shape = _lib.AttnShape(1, 61, 32, 2048)
    assert lib.tsv_tree_verify_attn_workspace_size(ctypes.byref(shape), ctypes.byref(cache)) == 0
    cache.head_dim = 128
    shape.num_q_heads = 30
    assert lib.tsv_tree_verify_attn(ctypes.byref(shape), p, p, p, ctypes.byref(cache), p, p, p, p,
                                    1e4, 0.1, p, None, 0, None, None) == 1
    shape.num_q_heads = 32
    assert lib.tsv_tree_verify_attn_workspace_size(ctypes.byref(shape), ctypes.byref(cache)) > 0
    # prep, attention and (when the keys are split) the merge
    assert lib.tsv_tree_verify_attn_launches(ctypes.byref(shape), ctypes.byref(cache)) in (2, 3)
    assert lib.tsv_tree_verify_attn(ctypes.byref(shape), p, p, p, ctypes.byref(cache), p, p, p, p,
                                    1e4, 0.1, p, None, 0, None, None) == 3
    # accept: contiguous capacity not a multiple of 64
    cache.capacity = 100
    assert lib.tsv_accept_and_compact(p, p, p, p, p, p, None, 1, 61, 7, ctypes.byref(cache),
                                      p, p, p, p, p, None, None) == 1
    # lm_head argmax: hidden size not a multiple of 64, negative rows, misaligned input,
    # workspace sizing (one 64-bit key per vocabulary range and row)
    assert lib.tsv_lm_head_argmax(p, p, 61, 96, 128256, p, None, p, 1 << 20, None) == 1
    assert lib.tsv_lm_head_argmax(p, p, -1, 4096, 128256, p, None, p, 1 << 20, None) == 1
    assert lib.tsv_lm_head_argmax(ctypes.c_void_p(24), p, 61, 4096, 128256, p, None, p,
                                  1 << 20, None) == 1
    assert lib.tsv_lm_head_argmax_workspace_size(-1, 100) == 0
    assert lib.tsv_lm_head_argmax_workspace_size(61, 0) == 0
    ws = lib.tsv_lm_head_argmax_workspace_size(61, 128256)
    assert ws > 0 and ws % 256 == 0 and ws >= 61 * 8


def test_host_validation_of_the_wider_calls(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: the checks fail first
    a256 = ctypes.c_void_p(4096)
    # non-greedy acceptance: vocab out of range, max_nodes out of range, small workspace
    args = lambda vocab, t, ws_bytes: ([p, None, vocab] + [p] * 12 + [1, t, 7, None] +
                                       [p] * 5 + [None, a256, ws_bytes, None])
    assert lib.tsv_tree_sample_accept(*args(0, 61, 1 << 20)) == 1
    assert lib.tsv_tree_sample_accept(*args((1 << 20) + 1, 61, 1 << 20)) == 1
    assert lib.tsv_tree_sample_accept(*args(1000, 257, 1 << 20)) == 1
    assert lib.tsv_tree_sample_accept(*args(1000, 61, 8)) == 3
    assert lib.tsv_tree_sample_accept_workspace_size(2, 61) >= 2 * 61 * 24
    assert lib.tsv_tree_sample_accept_workspace_size(2, 0) == 0
    assert lib.tsv_target_probs(p, 1000, p, p, p, p, p, 1, 61, p, a256, 8, None) == 3
    # fixed level: width above the limit, nodes past max_nodes, frontier overlapping
    assert lib.tsv_draft_fixed_level(p, 1, 2, 100, 100, 17, 3, 1, 64, p, p, None) == 1
    assert lib.tsv_draft_fixed_level(p, 1, 2, 100, 100, 4, 3, 1, 10, p, p, None) == 1
    assert lib.tsv_draft_fixed_level(p, 1, 3, 100, 100, 2, 3, 1, 64, p, p, None) == 1
    assert lib.tsv_draft_fixed_level(p, 1, 2, 50, 100, 2, 3, 1, 64, p, p, None) == 1
    # grown mask: new nodes past max_nodes, first_new 0
    assert lib.tsv_draft_grow_mask(p, p, p, p, 1, 60, 8, 64, None, None) == 1
    assert lib.tsv_draft_grow_mask(p, p, p, p, 1, 0, 4, 64, None, None) == 1
    # d2t: empty table
    assert lib.tsv_draft_to_target(p, p, 1, 61, p, 0, None, None) == 1
    # product expansion: the same checks as the log-score one
    assert lib.tsv_draft_topk_expand_product(p, 1, 1, 100, 100, 17, 1, None, None, 100,
                                             p, p, p, p, p, p, p, 1 << 20, None) == 1


def test_empty_batch_is_a_no_op(lib):
    assert lib.tsv_tree_sample_accept(*([None] * 2 + [1000] + [None] * 12 + [0, 61, 7, None] +
                                        [None] * 6 + [None, 0, None])) == 0
    assert lib.tsv_draft_fixed_level(None, 0, 2, 100, 100, 2, 3, 1, 64, None, None, None) == 0
    assert lib.tsv_draft_grow_mask(None, None, None, None, 0, 1, 4, 64, None, None) == 0
    assert lib.tsv_draft_to_target(None, None, 0, 61, None, 10, None, None) == 0
    assert lib.tsv_lm_head_argmax(None, None, 0, 64, 10, None, None, None, 0, None) == 0
    assert lib.tsv_tree_build_meta(None, None, None, 0, 8, 3, None, None, None, None, None,
                                   None, None, None) == 0


def test_lm_head_vocabulary_split_planner(lib):
    """The host planner of the lm-head kernel (no GPU here: the SM count reads as 148):
    one 64-bit key per (vocabulary range, row); the ranges are whole 32-entry chunks and
    their count minimises waves x (chunks per range + 1), the largest count on ties."""
    def model(rows, vocab, sms=148):
        m = -(-rows // 128)
        c = -(-vocab // 32)
        best = None
        for s in range(1, min(c, 8 * sms) + 1):
            cost = -(-(m * s) // sms) * (-(-c // s) + 1)
            if best is None or cost <= best[0]:
                best = (cost, s)
        return best[1]
    for rows, vocab in [(61, 128256), (976, 128256), (4160, 128256), (1, 1), (300, 30001)]:
        splits = model(rows, vocab)
        want = (splits * rows * 8 + 255) // 256 * 256
        assert lib.tsv_lm_head_argmax_workspace_size(rows, vocab) == want, (rows, vocab)


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_header_is_plain_c(tmp_path, lang, std):
    """include/tsv.h is a C header (no torch or CUDA types in the signatures): it compiles
    alone as C99 and as C++11 with warnings as errors."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("t.c" if lang == "c" else "t.cc")
    src.write_text('#include "tsv.h"\nint main(void) { return TSV_OK; }\n')
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", os.path.dirname(HEADER), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_attention_entry_points_share_host_checks(lib):
    """tsv_tree_verify_attn and tsv_tree_verify_attn_noalloc run one host validator: the
    same invalid arguments give the same status from both (every case below returns
    before any CUDA work)."""
    p = ctypes.c_void_p(16)
    k = ctypes.c_void_p(256)

    def both(shape, cache, q=p, mask=p, theta=1e4, scale=0.1):
        a = lib.tsv_tree_verify_attn(ctypes.byref(shape), q, p, p, ctypes.byref(cache), p, p, p,
                                     mask, theta, scale, p, p, 1 << 30, None, None)
        b = lib.tsv_tree_verify_attn_noalloc(ctypes.byref(shape), q, p, p, ctypes.byref(cache),
                                             p, p, p, mask, theta, scale, p, None, None)
        return a, b

    def fresh():
        return (_lib.AttnShape(2, 61, 32, 2048),
                _lib.KVCacheDesc(k, k, 1, 8, 128, 0, 2176, None, 0, 0, 1, 0))

    cases = []
    s, c = fresh(); c.head_dim = 96; cases.append(both(s, c))            # head_dim
    s, c = fresh(); s.num_q_heads = 30; cases.append(both(s, c))         # GQA mismatch
    s, c = fresh(); s.max_nodes = 257; cases.append(both(s, c))          # too many nodes
    s, c = fresh(); s.batch = 70000; cases.append(both(s, c))            # grid limit
    s, c = fresh(); c.capacity = 100; cases.append(both(s, c))           # capacity % 64
    s, c = fresh(); c.layout = 5; cases.append(both(s, c))               # unknown layout
    s, c = fresh(); c.layout = 1; cases.append(both(s, c))               # paged, no table
    s, c = fresh(); cases.append(both(s, c, theta=0.0))                  # RoPE theta
    s, c = fresh(); cases.append(both(s, c, scale=float("nan")))         # softmax scale
    s, c = fresh(); cases.append(both(s, c, q=ctypes.c_void_p(24)))      # misaligned q
    s, c = fresh(); cases.append(both(s, c, mask=None))                  # missing mask
    for a, b in cases:
        assert a == b == 1, cases
    s, c = fresh(); s.batch = 0
    assert both(s, c) == (0, 0)  # an empty batch is a no-op for both

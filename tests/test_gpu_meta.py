"""tsv_tree_build_meta vs the oracle, bit-exact, through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import tree
from tests import gpu_cases as gc
from tests.golden_io import load

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tree_speculative_decoding_verify_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def run_meta(parents_list, prefix, max_nodes, max_depth):
    import tree_speculative_decoding_verify_gb300 as T
    b = len(parents_list)
    par = np.full((b, max_nodes), -1, dtype=np.int32)
    nn = np.zeros(b, dtype=np.int32)
    for i, p in enumerate(parents_list):
        par[i, :len(p)] = p
        nn[i] = len(p)
    w = (max_nodes + 31) // 32
    d = gc.dev()
    o = dict(mask=torch.full((b, max_nodes, w), 7, dtype=torch.int32, device=d),
             position_ids=torch.full((b, max_nodes), 7, dtype=torch.int32, device=d),
             retrieve_indices=torch.full((b, max_nodes, max_depth + 1), 7, dtype=torch.int32,
                                         device=d),
             num_leaves=torch.full((b,), 7, dtype=torch.int32, device=d),
             next_token=torch.full((b, max_nodes), 7, dtype=torch.int32, device=d),
             next_sibling=torch.full((b, max_nodes), 7, dtype=torch.int32, device=d),
             err=torch.full((b,), 7, dtype=torch.int32, device=d))
    T.tree_build_meta(gc.i32(par), gc.i32(nn), gc.i32(prefix), max_depth, **o)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


def expect(parents, prefix, max_nodes, max_depth):
    p = list(int(x) for x in parents)
    n = len(p)
    w = (max_nodes + 31) // 32
    mask = np.zeros((max_nodes, w), dtype=np.uint32)
    mask[:n] = tree.pack_mask(tree.tree_mask(p), w)
    pos = np.full(max_nodes, prefix, dtype=np.int64)
    pos[:n] = tree.position_ids(p, prefix)
    ret = np.full((max_nodes, max_depth + 1), -1, dtype=np.int32)
    r = tree.retrieve_indices(p, max_depth + 1)
    ret[:len(r)] = r
    nxt = np.full(max_nodes, -1, dtype=np.int32)
    sib = np.full(max_nodes, -1, dtype=np.int32)
    a, s = tree.next_links(p)
    nxt[:n], sib[:n] = a, s
    return dict(mask=mask.view(np.int32), position_ids=pos.astype(np.int32),
                retrieve_indices=ret, num_leaves=len(r), next_token=nxt, next_sibling=sib)


def check(parents_list, prefix, max_nodes, max_depth):
    got = run_meta(parents_list, prefix, max_nodes, max_depth)
    for b, p in enumerate(parents_list):
        want = expect(p, int(prefix[b]), max_nodes, max_depth)
        assert got["err"][b] == 0
        for key in ("mask", "position_ids", "retrieve_indices", "next_token", "next_sibling"):
            np.testing.assert_array_equal(got[key][b], want[key], err_msg=f"{key} request {b}")
        assert got["num_leaves"][b] == want["num_leaves"]


def test_page_trees():
    g6 = load("six_node_mask.txt")["parents"]
    g221 = load("tree_221.txt")
    got = run_meta([g221["parents"]], [32], 11, 3)
    assert got["mask"][0][:, 0].astype(np.uint32).tolist() == g221["mask_words"]
    assert got["retrieve_indices"][0][:4].tolist() == g221["retrieve"]
    check([g6, g221["parents"]], np.array([5, 32]), 11, 4)


def test_dynamic_trees_of_every_workload():
    for name in ("llama8b", "long70b"):
        w = W.WORKLOADS[name]
        tok, par, _ = gc.oracle_tree(w, 0)
        check([par], np.array([w.max_prefix]), w.num_nodes, w.depth + 1)


@pytest.mark.parametrize("n,max_nodes", [(1, 1), (2, 33), (33, 40), (64, 64), (65, 96),
                                         (200, 256), (256, 256)])
def test_random_trees_span_mask_words(n, max_nodes):
    rng = np.random.default_rng(n)
    trees = [gc.random_tree(rng, int(rng.integers(1, n + 1)), 12) for _ in range(5)]
    trees[0] = gc.random_tree(rng, n, 12)
    check(trees, rng.integers(0, 5000, size=5), max_nodes, 12)


def test_chain_and_kary_and_fixed_branching():
    trees = [tree.kary_parents(17, 1), tree.kary_parents(40, 3),
             tree.fixed_branching_parents([2, 2, 1, 1]), tree.fixed_branching_parents([3, 3, 2])]
    check([np.array(t) for t in trees], np.array([0, 1, 2, 3]), 64, 16)


def test_bad_trees_report_errors_and_root_only_state():
    trees = [np.array([0, 0]), np.array([-1, 1, 0]), np.array([-1, 0, 1, 2, 3, 4])]
    got = run_meta(trees, np.array([10, 10, 10]), 8, 3)
    assert got["err"].tolist() == [1, 2, 3]
    for b in range(3):
        rows = got["mask"][b][:, 0].astype(np.uint32)
        assert rows.tolist() == [1 << i for i in range(8)]
        assert got["position_ids"][b].tolist() == [10] * 8
        assert got["num_leaves"][b] == 1
        assert got["retrieve_indices"][b][0].tolist() == [0, -1, -1, -1]
        assert (got["retrieve_indices"][b][1:] == -1).all()
        assert (got["next_token"][b] == -1).all() and (got["next_sibling"][b] == -1).all()


def test_bad_sizes():
    import tree_speculative_decoding_verify_gb300 as T
    d = gc.dev()
    b, t = 2, 4
    out = dict(mask=torch.zeros(b, t, 1, dtype=torch.int32, device=d),
               position_ids=torch.zeros(b, t, dtype=torch.int32, device=d),
               retrieve_indices=torch.zeros(b, t, 3, dtype=torch.int32, device=d),
               num_leaves=torch.zeros(b, dtype=torch.int32, device=d),
               next_token=torch.zeros(b, t, dtype=torch.int32, device=d),
               next_sibling=torch.zeros(b, t, dtype=torch.int32, device=d),
               err=torch.zeros(b, dtype=torch.int32, device=d))
    par = gc.i32([[-1, 0, 0, 1], [-1, 0, 0, 1]])
    T.tree_build_meta(par, gc.i32([5, 0]), gc.i32([3, 3]), 2, **out)
    assert out["err"].cpu().tolist() == [4, 4]
    T.tree_build_meta(par, gc.i32([4, 4]), gc.i32([-1, 3]), 2, **out)
    assert out["err"].cpu().tolist() == [4, 0]

"""Pins for the oracle's tree metadata: the pages' worked examples and invariants."""
import numpy as np
import pytest

from oracle import tree
from tests.golden_io import load, load_counts


def test_six_node_mask_matches_printed_example():
    g = load("six_node_mask.txt")
    mask = tree.tree_mask(g["parents"])
    assert mask.astype(int).tolist() == g["mask"]


def test_tree_221_diagram():
    g = load("tree_221.txt")
    parents = g["parents"]
    tree.validate_parents(parents)
    assert tree.tree_mask(parents).astype(int).tolist() == g["mask"]
    assert tree.depths(parents) == g["depths"]
    words = tree.pack_mask(tree.tree_mask(parents))
    assert words[:, 0].tolist() == g["mask_words"]
    assert tree.retrieve_indices(parents, 4).tolist() == g["retrieve"]
    nxt, sib = tree.next_links(parents)
    assert nxt.tolist() == g["next_token"]
    assert sib.tolist() == g["next_sibling"]


def test_tree_221_is_the_fixed_branching_tree():
    g = load("tree_221.txt")
    assert tree.fixed_branching_parents([2, 2, 1]) == g["parents"]


@pytest.mark.parametrize("branching,count", load_counts("node_counts.txt"))
def test_node_counts(branching, count):
    parents = tree.fixed_branching_parents(branching)
    tree.validate_parents(parents)
    assert len(parents) - 1 == count


def test_positions_siblings_share_and_root_is_prefix():
    parents = load("tree_221.txt")["parents"]
    pos = tree.position_ids(parents, 32)
    assert pos[0] == 32
    kids = tree.children_of(parents)
    for sibs in kids:
        assert len({int(pos[s]) for s in sibs}) <= 1
    for i in range(1, len(parents)):
        assert pos[i] == pos[parents[i]] + 1


def test_chain_mask_is_causal():
    parents = tree.kary_parents(9, 1)
    assert parents == [-1, 0, 1, 2, 3, 4, 5, 6, 7]
    mask = tree.tree_mask(parents)
    assert np.array_equal(mask, np.tril(np.ones((9, 9), dtype=bool)))
    assert tree.depths(parents) == list(range(9))


def test_kary_tree():
    parents = tree.kary_parents(13, 3)
    assert parents[1:4] == [0, 0, 0] and parents[4:7] == [1, 1, 1] and parents[12] == 3
    assert tree.depths(parents)[-1] == 2


def test_mask_row_counts_equal_depth_plus_one():
    rng = np.random.default_rng(1)
    for n in (1, 2, 5, 40, 70, 200):
        parents = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
        mask = tree.tree_mask(parents)
        d = tree.depths(parents)
        assert mask.sum(axis=1).tolist() == [x + 1 for x in d]
        assert np.array_equal(mask, np.tril(mask))  # ancestors precede


def test_pack_mask_spans_several_words():
    parents = tree.kary_parents(70, 1)   # row 69 sees 70 columns -> 3 words
    words = tree.pack_mask(tree.tree_mask(parents))
    assert words.shape == (70, 3)
    assert words[69].tolist() == [0xFFFFFFFF, 0xFFFFFFFF, 0x3F]
    assert words[31].tolist() == [0xFFFFFFFF, 0, 0]
    assert words[32].tolist() == [0xFFFFFFFF, 1, 0]


def test_retrieve_rows_are_root_to_leaf_paths():
    rng = np.random.default_rng(2)
    for n in (1, 3, 17, 61):
        parents = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
        cols = max(tree.depths(parents)) + 1
        r = tree.retrieve_indices(parents, cols)
        assert r.shape[0] == len(tree.leaves(parents))
        for row in r:
            row = [x for x in row if x >= 0]
            assert row[0] == 0
            for a, b in zip(row, row[1:]):
                assert parents[b] == a
            assert not tree.children_of(parents)[row[-1]]


def test_root_only_tree():
    assert tree.tree_mask([-1]).tolist() == [[True]]
    assert tree.retrieve_indices([-1], 3).tolist() == [[0, -1, -1]]
    nxt, sib = tree.next_links([-1])
    assert nxt.tolist() == [-1] and sib.tolist() == [-1]


@pytest.mark.parametrize("bad", [[0], [-1, 1], [-1, 0, 2], [-1, -1], [-1, 0, 5]])
def test_invalid_parents_rejected(bad):
    with pytest.raises(ValueError):
        tree.validate_parents(bad)


def test_grown_level_masks_equal_the_ancestor_mask():
    """Growing the drafter's mask level by level (the block construction) gives the
    ancestor mask and positions of the whole tree at every level; old rows never see new
    nodes."""
    from oracle import tree as Tr
    rng = np.random.default_rng(2)
    k, levels, prefix = 4, 5, 37
    parents = [-1]
    mask, pos = np.ones((1, 1), dtype=bool), np.array([prefix])
    frontier = [0]
    for _ in range(levels):
        new_par = [frontier[int(rng.integers(0, len(frontier)))] for _ in range(k)]
        n0 = len(parents)
        mask, pos = Tr.grow_level_mask(mask, pos, new_par)
        parents += new_par
        assert (mask == Tr.tree_mask(parents)).all()
        assert pos.tolist() == Tr.position_ids(parents, prefix).tolist()
        assert not mask[:n0, n0:].any()
        frontier = list(range(n0, n0 + k))

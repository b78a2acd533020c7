"""Pins for the oracle's acceptance and compaction: the two pages' acceptance rules
agree, brute force over all root-down paths, and a byte comparison of the cache."""
import numpy as np
import pytest

from oracle import accept, tree


def random_tree(rng, n, vocab=6):
    parents = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
    tokens = [int(rng.integers(0, vocab))]
    for i in range(1, n):
        sib = {tokens[j] for j in range(1, i) if parents[j] == parents[i]}
        free = [t for t in range(vocab + len(sib)) if t not in sib]
        tokens.append(int(free[int(rng.integers(0, len(free)))]))  # distinct among siblings
    return parents, tokens


def brute_longest(tokens, parents, target):
    """Longest root-down path where every step's token equals the parent's target."""
    best = [0]
    for leaf in range(len(tokens)):
        chain, j = [], leaf
        while j != -1:
            chain.append(j)
            j = parents[j]
        chain.reverse()
        ok = all(tokens[b] == target[a] for a, b in zip(chain, chain[1:]))
        if ok and len(chain) > len(best):
            best = chain
    return best


@pytest.mark.parametrize("seed", range(60))
def test_walk_equals_posterior_and_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    parents, tokens = random_tree(rng, n, vocab=5)
    target = [int(rng.integers(0, 5)) for _ in range(n)]
    path, bonus = accept.greedy_walk(tokens, parents, target)
    assert path == brute_longest(tokens, parents, target)
    assert bonus == target[path[-1]]
    cols = max(tree.depths(parents)) + 1
    retrieve = tree.retrieve_indices(parents, cols)
    row, acc = accept.evaluate_posterior(tokens, retrieve, target)
    assert acc + 1 == len(path)
    assert [x for x in retrieve[row][:acc + 1]] == path


def test_walk_on_the_221_tree():
    parents = [-1, 0, 0, 1, 1, 2, 2, 3, 4, 5, 6]
    tokens = [9, 10, 11, 12, 13, 14, 15, 16, 17, 18, 19]
    target = [11, 0, 15, 0, 0, 0, 19, 0, 0, 0, 42]   # root -> B1 -> B2' -> B3'
    path, bonus = accept.greedy_walk(tokens, parents, target)
    assert path == [0, 2, 6, 10] and bonus == 42
    target[0] = 99                                     # nothing accepted
    assert accept.greedy_walk(tokens, parents, target) == ([0], 99)


def test_compaction_moves_rows_and_keeps_the_rest():
    rng = np.random.default_rng(0)
    cache = rng.normal(size=(2, 3, 20, 4))             # [layers, heads, slots, D]
    p_len, path = 7, [0, 2, 3, 9]                      # overlapping source/destination
    out = accept.compact(cache, p_len, path)
    for i, n in enumerate(path):
        assert np.array_equal(out[:, :, p_len + i], cache[:, :, p_len + n])
    untouched = [s for s in range(20) if not p_len <= s < p_len + len(path)]
    assert np.array_equal(out[:, :, untouched], cache[:, :, untouched])
    assert accept.slot_map(p_len, path) == [(7, 7), (9, 8), (10, 9), (16, 10)]


def test_compaction_matches_sequential_copy_order():
    rng = np.random.default_rng(1)
    for _ in range(20):
        parents, tokens = random_tree(rng, 15, vocab=3)
        target = [int(rng.integers(0, 3)) for _ in range(15)]
        path, _ = accept.greedy_walk(tokens, parents, target)
        cache = rng.normal(size=(30, 2))
        seq = cache.copy()
        for i, n in enumerate(path):                    # increasing i is safe: path[i] >= i
            seq[5 + i] = seq[5 + n]
        assert np.array_equal(accept.compact(cache, 5, path), seq)


def test_every_valid_path_is_reachable_by_some_target():
    parents = [-1, 0, 0, 1, 1, 2]
    tokens = [0, 1, 2, 3, 4, 5]
    for node in range(6):
        chain, j = [], node
        while j != -1:
            chain.append(j)
            j = parents[j]
        chain.reverse()
        target = [7] * 6
        for a, b in zip(chain, chain[1:]):
            target[a] = tokens[b]
        assert accept.greedy_walk(tokens, parents, target)[0] == chain


def test_request_without_a_tree_accepts_the_root_only():
    """A released slot (tree_valid false) takes the single-token path even where the
    target would accept a child: path [0], bonus = the target's argmax at the root."""
    parents = [-1, 0, 0, 1]
    tokens = [5, 7, 8, 9]
    target = [7, 9, 3, 4]  # with a tree: 0 -> 1 -> 3
    assert accept.greedy_walk(tokens, parents, target) == ([0, 1, 3], 4)
    assert accept.greedy_walk(tokens, parents, target, tree_valid=False) == ([0], 7)

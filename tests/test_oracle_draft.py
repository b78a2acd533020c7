"""Pins for the oracle's dynamic tree expansion: closed forms, brute force, the pages'
counts and the invariants of the selection."""
import math

import numpy as np
import pytest

from oracle import draft, tree

F32 = np.float32


def brute_topk(values, k):
    """Rank by counting: rank(i) = #{j : v_j > v_i or (v_j == v_i and j < i)}."""
    v = [float(x) for x in values]
    rank = [sum(1 for j in range(len(v)) if v[j] > v[i] or (v[j] == v[i] and j < i))
            for i in range(len(v))]
    return [i for r in range(k) for i in range(len(v)) if rank[i] == r]


def test_logsumexp_closed_forms():
    assert math.isclose(draft.logsumexp(np.full(7, 3.0)), 3.0 + math.log(7), rel_tol=1e-15)
    a, b = 1.25, -0.5
    assert math.isclose(draft.logsumexp([a, b]), math.log(math.exp(a) + math.exp(b)),
                        rel_tol=1e-15)
    big = np.array([1000.0, 1000.0])          # overflow-safe by the max shift
    assert math.isclose(draft.logsumexp(big), 1000.0 + math.log(2.0), rel_tol=1e-15)
    lp = draft.log_softmax(np.random.default_rng(0).normal(0, 2, 500))
    assert math.isclose(float(np.exp(lp).sum()), 1.0, rel_tol=1e-12)


@pytest.mark.parametrize("seed", range(20))
def test_row_topk_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    x = rng.integers(-3, 4, size=9).astype(F32)   # many exact ties
    k = int(rng.integers(1, 9))
    assert draft.row_topk(x, k).tolist() == brute_topk(x, k)


@pytest.mark.parametrize("seed", range(10))
def test_topk_by_score_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    s = (rng.integers(-4, 4, size=25) * 0.5).astype(F32)
    assert draft.topk_by_score(s, 6) == brute_topk(s, 6)


def test_candidate_count_matches_both_pages():
    for k, depth in [(10, 6), (8, 7), (3, 2), (1, 5)]:
        levels = depth + 1                        # [TRT]: D draft levels
        assert draft.num_candidates(k, depth) == k + k * k * (levels - 1)
    assert draft.num_candidates(10, 6) == 610
    assert draft.num_candidates(8, 7) == 456


def make_levels(seed, k, depth, v, sigma=2.0):
    rng = np.random.default_rng(seed)
    out = [rng.normal(0, sigma, (1, v)).astype(F32)]
    out += [rng.normal(0, sigma, (k, v)).astype(F32) for _ in range(depth)]
    return out


@pytest.mark.parametrize("k,depth,v", [(3, 2, 40), (4, 3, 64), (10, 2, 300)])
def test_expansion_structure_and_brute_force(k, depth, v):
    levels = make_levels(k * 7 + depth, k, depth, v)
    exp = draft.topk_generate(levels, k)
    assert exp.store_token.size == draft.num_candidates(k, depth)
    for li, lv in enumerate(exp.levels):
        lg = levels[li]
        r = lg.shape[0]
        # per-row: tokens are the row's brute-force top-k, logp = x - lse
        for s in range(r):
            assert lv.tokens[s * k:(s + 1) * k].tolist() == brute_topk(lg[s], k)
            lse = draft.logsumexp(lg[s])
            for c in range(k):
                t = lv.tokens[s * k + c]
                assert lv.logp[s * k + c] == F32(float(lg[s, t]) - lse)
                assert lv.logp[s * k + c] <= 0
        # joint selection = brute-force top-k of the fp32 cumulative scores
        assert lv.selected == brute_topk(lv.cu, k)


@pytest.mark.parametrize("seed", range(4))
def test_store_score_is_path_sum_of_logp(seed):
    """Every candidate's score is the fp32 running sum of log-probabilities along its
    ancestor chain, root first: an independent walk of the parent links."""
    k, depth = 4, 3
    levels = make_levels(50 + seed, k, depth, 80)
    exp = draft.topk_generate(levels, k)
    logp = np.concatenate([lv.logp for lv in exp.levels])
    for c in range(exp.store_token.size):
        chain = []
        j = c
        while j != -1:
            chain.append(j)
            j = int(exp.store_parent[j])
        acc = F32(0.0)
        for j in reversed(chain):
            acc = F32(acc + logp[j])
        assert exp.store_score[c] == acc
        # the parent of a level-l candidate is a selected node of level l-1
        assert len(chain) == 1 + sum(c >= draft.level_store_offset(lv, k)
                                     for lv in range(2, depth + 2))


def test_parent_of_flat_index_is_flat_div_k():
    k, depth = 3, 2
    levels = make_levels(7, k, depth, 30)
    exp = draft.topk_generate(levels, k)
    prev = exp.levels[0]
    front_store = [draft.level_store_offset(1, k) + f for f in prev.selected]
    lv = exp.levels[1]
    for flat in range(k * k):
        assert lv.parent_store[flat] == front_store[flat // k]


@pytest.mark.parametrize("k,depth,total", [(3, 2, 5), (4, 3, 20), (10, 6, 60), (8, 7, 48)])
def test_final_selection_invariants(k, depth, total):
    levels = make_levels(k + depth + total, k, depth, 200)
    exp = draft.topk_generate(levels, k)
    tokens, parents = draft.select_final(exp.store_token, exp.store_score, exp.store_parent,
                                         total, 77)
    assert tokens.size == total + 1 and tokens[0] == 77
    tree.validate_parents(parents.tolist())
    best = brute_topk(exp.store_score, total)
    chosen = sorted(best)
    assert tokens[1:].tolist() == [int(exp.store_token[c]) for c in chosen]
    for i, c in enumerate(chosen):
        p = int(exp.store_parent[c])
        assert parents[i + 1] == (0 if p < 0 else chosen.index(p) + 1)
    # scores never increase from parent to child
    for i in range(2, total + 1):
        c, p = chosen[i - 1], parents[i]
        if p > 0:
            assert exp.store_score[c] <= exp.store_score[chosen[p - 1]]


def test_exact_ties_take_lower_indices():
    k, v = 2, 6
    row = np.array([[1.0, 3.0, 3.0, 0.0, 3.0, -1.0]], dtype=F32)
    lv = draft.expand_level(row, k)
    assert lv.tokens.tolist() == [1, 2]                # three-way tie at 3.0
    rows = np.array([[0.0, 2.0, 1.0, 0.0, 0.0, 0.0]] * 2, dtype=F32)  # duplicate rows
    lv2 = draft.expand_level(rows, k, np.array([-1.0, -1.0], F32), np.array([0, 1], np.int32))
    assert lv2.cu[0] == lv2.cu[2] and lv2.selected == [0, 2]
    assert v == row.shape[1]


def test_total_tokens_equal_to_store_keeps_everything():
    k, depth = 2, 2
    levels = make_levels(3, k, depth, 20)
    exp = draft.topk_generate(levels, k)
    c = draft.num_candidates(k, depth)
    tokens, parents = draft.select_final(exp.store_token, exp.store_score, exp.store_parent, c, 5)
    assert tokens[1:].tolist() == exp.store_token.tolist()
    assert parents[1:k + 1].tolist() == [0] * k

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


# ---- expansion variants ------------------------------------------------------------
def test_product_scores_are_the_exponentials_of_the_log_sums():
    """[TRT]'s parent-times-child probability scores: each equals exp of the log-domain
    cumulative score (within fp32 rounding), so both modes rank alike wherever the log
    scores are apart."""
    from oracle import draft as D
    rng = np.random.default_rng(4)
    k, depth, v = 4, 3, 60
    levels = [rng.normal(0, 2, (1, v)).astype(np.float32)] + \
        [rng.normal(0, 2, (k, v)).astype(np.float32) for _ in range(depth)]
    lg = D.topk_generate(levels, k)
    pr = D.topk_generate(levels, k, product=True)
    np.testing.assert_allclose(pr.store_score, np.exp(lg.store_score.astype(np.float64)),
                               rtol=1e-5)
    if D.margins(lg, 8) > 1e-4:
        for a, b in zip(lg.levels, pr.levels):
            assert a.selected == b.selected
    assert lg.store_token.tolist() == pr.store_token.tolist()
    assert lg.store_parent.tolist() == pr.store_parent.tolist()
    # the base layer's product scores are the top-k probabilities themselves
    p = np.exp(levels[0][0].astype(np.float64) - np.log(np.exp(levels[0][0].astype(np.float64)).sum()))
    np.testing.assert_allclose(pr.store_score[:k], np.sort(p)[::-1][:k], rtol=1e-6)


def test_draft_to_target_map():
    from oracle import draft as D
    toks = np.array([77, 0, 3, 5, 9, 2], np.int32)
    ident = np.arange(8)
    assert D.map_draft_to_target(toks, 6, ident).tolist() == [77, 0, 3, 5, -1, 2]
    perm = np.array([10, 11, 12, 13, 14, 15, 16, 17]) * 3
    assert D.map_draft_to_target(toks, 4, perm).tolist() == [77, 30, 39, 45, 9, 2]


def test_fixed_tree_by_hand_and_by_property():
    from oracle import draft as D
    from oracle import tree as Tr
    root_row = np.array([[0.1, 0.9, 0.5, 0.9, -1.0]], np.float32)  # tie: id 1 before 3
    lvl2 = np.array([[5, 0, 0, 0, 0], [0, 0, 0, 0, 2]], np.float32)
    tokens, parents = D.fixed_tree([root_row, lvl2], [2, 1], 42)
    assert tokens.tolist() == [42, 1, 3, 0, 4]
    assert parents.tolist() == [-1, 0, 0, 1, 2]
    rng = np.random.default_rng(9)
    branching = [3, 2, 2]
    frontier, rows = 1, []
    for wdt in branching:
        rows.append(rng.normal(size=(frontier, 40)).astype(np.float32))
        frontier *= wdt
    tokens, parents = D.fixed_tree(rows, branching, 7)
    assert parents.tolist() == Tr.fixed_branching_parents(branching)
    # every node's children carry its row's top tokens, best first
    depth = Tr.depths(parents.tolist())
    level_nodes = {}
    for i, d in enumerate(depth):
        level_nodes.setdefault(d, []).append(i)
    for d, nodes in level_nodes.items():
        if d >= len(branching):
            continue
        for f, node in enumerate(nodes):
            kids = [c for c in range(len(parents)) if parents[c] == node]
            row = rows[d][f]
            assert tokens[kids].tolist() == np.argsort(-row, kind="stable")[:branching[d]].tolist()

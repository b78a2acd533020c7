"""The non-greedy acceptance oracle against closed forms, special cases that reduce to
the greedy walk, and the output-distribution guarantee of rejection sampling."""
import numpy as np
import pytest

from oracle import accept, sampling

P4 = np.array([0.5, 0.3, 0.15, 0.05])
L4 = np.log(P4)


def test_temperature_scales_the_softmax():
    np.testing.assert_allclose(sampling.filter_probs(L4, 1.0), P4, rtol=1e-12)
    sq = P4 ** 2 / (P4 ** 2).sum()  # logits / 0.5 = 2 log p
    np.testing.assert_allclose(sampling.filter_probs(L4, 0.5), sq, rtol=1e-12)


def test_greedy_limits():
    lg = np.array([1.0, 3.0, 3.0, -2.0])
    for p in (sampling.filter_probs(lg, 0.0), sampling.filter_probs(lg, 0.7, top_k=1)):
        assert p.tolist() == [0.0, 1.0, 0.0, 0.0]  # the first maximum


def test_top_k_keeps_the_lower_id_on_a_tie():
    lg = np.array([2.0, 0.0, 1.0, 1.0])
    p = sampling.filter_probs(lg, 1.0, top_k=2)
    want = np.array([np.e, 0, 1, 0]) / (np.e + 1)
    np.testing.assert_allclose(p, want, rtol=1e-12)


@pytest.mark.parametrize("top_p,kept", [(0.49, [0]), (0.51, [0, 1]), (0.79, [0, 1]),
                                        (0.81, [0, 1, 2]), (0.0, [0]), (0.999, [0, 1, 2, 3])])
def test_top_p_keeps_the_token_that_crosses(top_p, kept):
    p = sampling.filter_probs(L4, 1.0, top_p=top_p)
    assert np.flatnonzero(p).tolist() == kept
    np.testing.assert_allclose(p[kept], P4[kept] / P4[kept].sum(), rtol=1e-12)


def test_top_p_applies_to_the_renormalised_top_k():
    # after top-3 the masses are [0.526, 0.316, 0.158]: the third has 0.842 before it
    assert np.flatnonzero(sampling.filter_probs(L4, 1.0, top_k=3, top_p=0.83)).tolist() == [0, 1]
    assert np.flatnonzero(sampling.filter_probs(L4, 1.0, top_k=3, top_p=0.85)).tolist() == [0, 1, 2]


@pytest.mark.parametrize("min_p,kept", [(0.25, [0, 1, 2]), (0.7, [0]), (0.09, [0, 1, 2, 3])])
def test_min_p_is_relative_to_the_largest(min_p, kept):
    p = sampling.filter_probs(L4, 1.0, min_p=min_p)
    assert np.flatnonzero(p).tolist() == kept
    np.testing.assert_allclose(p.sum(), 1.0, rtol=1e-12)


@pytest.mark.parametrize("u,t", [(0.0, 0), (0.1999, 0), (0.2, 2), (0.69, 2), (0.7, 3),
                                 (0.9999, 3)])
def test_inverse_cdf_skips_zero_mass(u, t):
    assert sampling.sample_inverse_cdf([0.2, 0.0, 0.5, 0.3], u) == t


def _random_tree(rng, n, vocab):
    parents = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
    tokens = [int(rng.integers(0, vocab))]
    for i in range(1, n):
        used = {tokens[j] for j in range(1, i) if parents[j] == parents[i]}
        free = [t for t in range(vocab) if t not in used]
        tokens.append(free[int(rng.integers(0, len(free)))])
    return tokens, parents


def test_zero_temperature_is_the_greedy_walk():
    rng = np.random.default_rng(1)
    for _ in range(200):
        n, vocab = int(rng.integers(1, 14)), 5
        tokens, parents = _random_tree(rng, n, vocab)
        logits = rng.normal(size=(n, vocab)).round(1)
        # plant a walk so that acceptances happen
        node = 0
        while True:
            kids = sampling.children(parents, node)
            if not kids or rng.random() < 0.3:
                break
            c = kids[int(rng.integers(0, len(kids)))]
            logits[node, tokens[c]] = 9.0
            node = c
        probs = [sampling.filter_probs(r, 0.0) for r in logits]
        target = [int(np.argmax(r)) for r in logits]
        got = sampling.rejection_walk(tokens, parents, probs, rng.random(n), rng.random())
        assert got == accept.greedy_walk(tokens, parents, target)
        probs1 = [sampling.filter_probs(r, 1.3, top_k=1) for r in logits]
        assert sampling.rejection_walk(tokens, parents, probs1, rng.random(n), rng.random()) == got


def test_invalid_tree_samples_at_the_root():
    probs = [np.array([0.2, 0.0, 0.5, 0.3])] * 3
    assert sampling.rejection_walk([1, 2, 3], [-1, 0, 0], probs, [0.0] * 3, 0.75,
                                   tree_valid=False) == ([0], 3)


def _first_token(tokens, parents, probs, u_node, u_final, q=None):
    path, tok = sampling.rejection_walk(tokens, parents, probs, u_node, u_final, q)
    return tokens[path[1]] if len(path) > 1 else tok


def _draw_without_replacement(rng, q, k):
    """k distinct tokens drawn one after another from q, each from what is left of q
    renormalised (successive sampling)."""
    rem, out = np.array(q, np.float64), []
    for _ in range(k):
        x = int(rng.choice(len(rem), p=rem / rem.sum()))
        out.append(x)
        rem[x] = 0.0
    return out


@pytest.mark.parametrize("mode", ["target_only", "draft_aware"])
def test_first_emitted_token_follows_the_target(mode):
    """The guarantee of rejection sampling: the first token the step emits (an accepted
    child's token, else the sample at the root) is distributed as the filtered target
    distribution at the root. Target-only holds for any fixed candidates; the
    draft-aware rule for distinct siblings drawn from q without replacement."""
    rng = np.random.default_rng(7)
    p_root = np.array([0.05, 0.4, 0.1, 0.3, 0.15])
    q_root = np.array([0.3, 0.1, 0.25, 0.05, 0.3])
    parents = [-1, 0, 0, 0, 1, 2]
    other = np.array([0.2, 0.2, 0.2, 0.2, 0.2])
    probs = [p_root] + [other] * 5
    n = 60000
    counts = np.zeros(5)
    for _ in range(n):
        if mode == "target_only":
            tokens, q = [0, 3, 0, 4, 1, 2], None
        else:
            tokens = [0] + _draw_without_replacement(rng, q_root, 3) + [1, 2]
            q = [q_root] + [other] * 5
        counts[_first_token(tokens, parents, probs, rng.random(6), rng.random(), q)] += 1
    freq = counts / n
    sigma = np.sqrt(p_root * (1 - p_root) / n)
    assert (np.abs(freq - p_root) < 4.5 * sigma).all(), (freq, p_root)


def _exact_first_token(p_root, cand, q_root=None):
    """The distribution of the first emitted token of a root with candidate children
    `cand`, integrated exactly over the uniforms: every accept/reject pattern is forced
    through the walk (u = 0 accepts, u just below 1 rejects) and weighted by the
    acceptance probabilities the walk's trace reports."""
    k = len(cand)
    tokens, parents = [0] + list(cand), [-1] + [0] * k
    probs = [p_root] * (k + 1)
    q = None if q_root is None else [q_root] * (k + 1)
    out = np.zeros(len(p_root))
    below_one = np.nextafter(1.0, 0.0)
    for stop in range(k + 1):  # accept candidate `stop`, or (stop == k) reject them all
        u = [below_one] * (k + 1)
        if stop < k:
            u[stop + 1] = 0.0
        trace = []
        path, _ = sampling.rejection_walk(tokens, parents, probs, u, 0.0, q, True, trace)
        tests = [a for kind, _, a in trace if kind == "test"]
        if len(tests) != min(stop + 1, k) or (len(path) > 1) != (stop < k):
            continue  # this pattern has probability zero (an acceptance of 0 or 1)
        w = np.prod([1.0 - a for a in tests[:stop]])
        if stop < k:
            out[tokens[path[1]]] += w * tests[stop]
        else:
            final = [d for kind, _, d in trace if kind == "final"][0]
            out += w * final / final.sum()
    return out


def test_first_token_distribution_is_exact_for_draws_without_replacement():
    """Integrated over every ordered draw of three distinct candidates from q (each
    draw's probability by successive sampling) and over the uniforms, the first emitted
    token is distributed exactly as p. The same holds for target-only on any fixed
    candidate list."""
    import itertools
    p_root = np.array([0.05, 0.4, 0.1, 0.3, 0.15])
    q_root = np.array([0.3, 0.1, 0.25, 0.05, 0.3])
    total = np.zeros(5)
    for seq in itertools.permutations(range(5), 3):
        pr, rem = 1.0, q_root.copy()
        for x in seq:
            pr *= rem[x] / rem.sum()
            rem[x] = 0.0
        total += pr * _exact_first_token(p_root, seq, q_root)
    np.testing.assert_allclose(total, p_root, atol=1e-12)
    for cand in ([3, 0, 4], [1], [4, 3, 2, 1, 0]):
        np.testing.assert_allclose(_exact_first_token(p_root, cand), p_root, atol=1e-12)


def test_rejected_tokens_are_never_the_correction():
    rng = np.random.default_rng(3)
    p = np.array([0.3, 0.3, 0.2, 0.2])
    tokens, parents = [9, 0, 1], [-1, 0, 0]
    for _ in range(2000):
        u = rng.random(3)
        path, tok = sampling.rejection_walk(tokens, parents, [p, p, p], u, rng.random())
        if path == [0]:
            assert tok not in (0, 1)


def test_degenerate_parameters():
    """min_p above 1 keeps the largest; a non-finite maximum or top_p <= 0 is greedy; NaN
    never wins."""
    assert sampling.filter_probs(L4, 1.0, min_p=3.0).tolist() == [1.0, 0.0, 0.0, 0.0]
    assert sampling.filter_probs(L4, 1.0, top_p=-0.5).tolist() == [1.0, 0.0, 0.0, 0.0]
    lg = np.array([0.0, np.inf, np.inf, 1.0])
    assert sampling.filter_probs(lg, 1.0).tolist() == [0.0, 1.0, 0.0, 0.0]
    lg = np.array([np.nan, -1.0, 2.0])
    assert sampling.filter_probs(lg, 0.0).tolist() == [0.0, 0.0, 1.0]
    assert np.isfinite(sampling.filter_probs(lg, 1.0)).all()
    assert sampling.filter_probs(np.full(3, -np.inf), 1.0).tolist() == [1.0, 0.0, 0.0]

"""The lm-head argmax oracle against constructions whose answer is known."""
import numpy as np

from oracle import lm_head


def test_planted_rows_win_by_a_margin():
    """Vocabulary row c_m = 3 h_m gives logit 3 |h_m|^2, far above every random row."""
    rng = np.random.default_rng(0)
    rows, hdim, v = 7, 96, 5000
    h = rng.standard_normal((rows, hdim))
    w = rng.standard_normal((v, hdim)) * 0.01
    plant = rng.choice(v, rows, replace=False)
    for m, c in enumerate(plant):
        w[c] = 3 * h[m]
    idx, best = lm_head.lm_head_argmax(h, w, chunk=1024)
    assert idx.tolist() == plant.tolist()
    np.testing.assert_allclose(best, 3 * (h * h).sum(axis=1), rtol=1e-12)


def test_ties_go_to_the_lower_index_across_chunks():
    """Three equal best rows, in different chunks: the first one is the answer."""
    h = np.ones((2, 4))
    w = np.zeros((3000, 4))
    for c in (2999, 1700, 900):
        w[c] = 1.0
    w[5, 0] = -1.0
    idx, best = lm_head.lm_head_argmax(h, w, chunk=1000)
    assert idx.tolist() == [900, 900]
    assert best.tolist() == [4.0, 4.0]


def test_negative_logits_and_a_single_entry():
    """All logits negative: the least negative wins; a one-entry vocabulary answers 0."""
    h = np.array([[1.0, -2.0]])
    w = np.array([[5.0, 5.0], [1.0, 1.0], [2.0, 3.0]])  # logits -5, -1, -4
    assert lm_head.lm_head_argmax(h, w)[0].tolist() == [1]
    assert lm_head.lm_head_argmax(h, w[:1])[0].tolist() == [0]

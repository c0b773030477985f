"""Pins for the oracle's top-k temperature sampler (ds4f-disk issue #6, work
item 3: the head's logits go to top-k / temperature sampling; step 3: a
softmax sampler driven by a seeded generator, equal seeds giving equal
tokens).

The selection is checked against Python's sort with an explicit key; the
probabilities against scipy's softmax, the two-entry logistic closed form
and equal-logit uniformity; the draw against the frequencies a fine grid of
u produces; and the limits (T = 0, NaN, +/-inf) against their definitions.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle


def sort_order(y):
    """Greedy order by sorting: NaN first, then the larger value, then the lower index."""
    return sorted(range(len(y)), key=lambda i: (0 if math.isnan(y[i]) else 1,
                                                 0.0 if math.isnan(y[i]) else -float(y[i]), i))


def test_selection_matches_sorted_with_ties_nans_infs_and_signed_zeros():
    rng = np.random.default_rng(31)
    for trial in range(300):
        n = int(rng.integers(1, 80))
        y = rng.integers(-4, 5, n).astype(np.float32)  # many ties
        if trial % 3 == 0:
            y[rng.integers(0, n, 3)] = np.nan
        if trial % 4 == 0:
            y[rng.integers(0, n, 2)] = np.inf
        if trial % 5 == 0:
            y[rng.integers(0, n, 2)] = -np.inf
        if trial % 7 == 0:
            y[rng.integers(0, n, 4)] = -0.0
        k = int(rng.integers(1, n + 1))
        idx, _, _ = oracle.topk_sample(y, k, 1.0, 0.5)
        assert list(idx[0]) == sort_order(y)[:k]


def test_probabilities_match_scipy_softmax():
    rng = np.random.default_rng(32)
    for T in (0.25, 0.7, 1.0, 3.0):
        y = (rng.standard_normal((3, 500)) * 4).astype(np.float32)
        k = 40
        idx, prob, _ = oracle.topk_sample(y, k, T, [0.1, 0.5, 0.9])
        for v in range(3):
            ref = softmax(y[v, idx[v]].astype(np.float64) / T)
            assert np.allclose(prob[v], ref, rtol=1e-12, atol=0)
            assert np.all(np.diff(prob[v]) <= 0)  # best first


def test_two_entries_logistic_closed_form():
    a, b, T = np.float32(1.75), np.float32(-0.5), 0.8
    _, prob, _ = oracle.topk_sample(np.array([b, a], np.float32), 2, T, 0.0)
    p0 = 1.0 / (1.0 + math.exp((float(b) - float(a)) / T))
    assert prob[0, 0] == pytest.approx(p0, rel=1e-15)
    assert prob[0, 1] == pytest.approx(1 - p0, rel=1e-14)


@pytest.mark.parametrize("k", [1, 2, 5, 64])
def test_equal_logits_are_uniform_and_u_picks_its_slot(k):
    y = np.full(100, 2.5, np.float32)
    for j in range(k):
        idx, prob, tok = oracle.topk_sample(y, k, 1.3, (j + 0.5) / k)
        assert list(idx[0]) == list(range(k))
        assert np.allclose(prob[0], 1.0 / k, rtol=1e-15)
        assert tok[0] == j


def test_token_frequencies_on_a_u_grid_equal_the_probabilities():
    rng = np.random.default_rng(33)
    y = (rng.standard_normal(300) * 2).astype(np.float32)
    k, T, N = 12, 0.9, 20000
    us = (np.arange(N) + 0.5) / N
    idx, prob, tok = oracle.topk_sample(np.tile(y, (N, 1)), k, T, us)
    counts = np.array([(tok == i).sum() for i in idx[0]])
    assert counts.sum() == N
    assert np.all(np.abs(counts - N * prob[0]) <= 1.0)
    # the draw is monotone in u: tokens come out in rank order along the grid
    rank = {int(i): r for r, i in enumerate(idx[0])}
    assert np.all(np.diff([rank[int(t)] for t in tok]) >= 0)


def test_shift_and_temperature_scaling_invariance():
    rng = np.random.default_rng(34)
    y = rng.integers(-50, 50, 400).astype(np.float32)  # exact under +16 and x2
    k = 30
    base = oracle.topk_sample(y, k, 1.5, 0.37)
    shifted = oracle.topk_sample(y + np.float32(16), k, 1.5, 0.37)
    scaled = oracle.topk_sample(y * np.float32(2), k, 3.0, 0.37)
    for other in (shifted, scaled):
        assert np.array_equal(base[0], other[0])
        assert np.array_equal(base[1], other[1])
        assert np.array_equal(base[2], other[2])


def test_temperature_zero_is_greedy_and_small_temperature_tends_to_it():
    rng = np.random.default_rng(35)
    y = rng.standard_normal((4, 1000)).astype(np.float32)
    for u in (0.0, 0.5, 0.999):
        idx, prob, tok = oracle.topk_sample(y, 8, 0.0, u)
        assert np.array_equal(tok, oracle.argmax_rows(y))
        assert np.array_equal(prob[:, 0], np.ones(4)) and not prob[:, 1:].any()
        _, prob_s, tok_s = oracle.topk_sample(y, 8, 1e-6, u)
        assert np.array_equal(tok_s, tok)
        assert np.all(prob_s[:, 0] > 1 - 1e-12)


def test_k_one_is_greedy_at_any_temperature():
    y = np.array([[0.5, 3.0, 3.0, -1.0]], np.float32)
    idx, prob, tok = oracle.topk_sample(y, 1, 2.0, 0.99)
    assert idx[0, 0] == 1 and tok[0] == 1 and prob[0, 0] == 1.0


def test_u_clamping():
    y = np.array([4.0, 1.0, 3.0, 2.0], np.float32)
    idx, _, _ = oracle.topk_sample(y, 4, 1.0, 0.0)
    assert list(idx[0]) == [0, 2, 3, 1]
    for u, want in ((0.0, 0), (-0.5, 0), (np.nan, 0), (1.0, 1), (7.0, 1)):
        assert oracle.topk_sample(y, 4, 1.0, u)[2][0] == want


def test_nonfinite_limits():
    # NaN best: entry 0, probabilities NaN
    y = np.array([1.0, np.nan, 5.0, np.nan], np.float32)
    idx, prob, tok = oracle.topk_sample(y, 3, 1.0, 0.7)
    assert list(idx[0]) == [1, 3, 2] and tok[0] == 1 and np.isnan(prob).all()
    # +inf entries share the weight; finite and -inf entries get none
    y = np.array([np.inf, 2.0, np.inf, -np.inf, np.inf], np.float32)
    idx, prob, tok = oracle.topk_sample(y, 5, 1.0, 0.5)
    assert list(idx[0]) == [0, 2, 4, 1, 3]
    assert np.allclose(prob[0], [1 / 3, 1 / 3, 1 / 3, 0, 0], rtol=1e-15)
    assert tok[0] == 2
    # a -inf entry below a finite best has probability 0 and is never drawn
    y = np.array([0.0, -np.inf, -1.0], np.float32)
    idx, prob, tok = oracle.topk_sample(y, 3, 1.0, 0.999999)
    assert list(idx[0]) == [0, 2, 1] and prob[0, 2] == 0.0 and tok[0] == 2
    # every entry -inf: equal weights
    y = np.full(6, -np.inf, np.float32)
    _, prob, tok = oracle.topk_sample(y, 4, 1.0, 0.6)
    assert np.allclose(prob[0], 0.25) and tok[0] == 2


def test_huge_logit_range_does_not_overflow():
    y = np.array([3e38, -3e38, 1e38], np.float32)
    _, prob, tok = oracle.topk_sample(y, 3, 1.0, 0.9)
    assert list(prob[0]) == [1.0, 0.0, 0.0] and tok[0] == 0


def test_rejects_bad_arguments():
    y = np.zeros((1, 5), np.float32)
    for k, T in ((0, 1.0), (6, 1.0), (2, -1.0), (2, float("nan"))):
        with pytest.raises(ValueError):
            oracle.topk_sample(y, k, T, 0.5)


def test_draw_intervals_are_closed_below_open_above():
    """Entry i owns u * S in [c_{i-1}, c_i): at an exact boundary the draw
    goes to the next entry (equal weights make the boundaries exact)."""
    y = np.zeros(10, np.float32)
    for k in (2, 4, 8):
        for j in range(1, k):
            assert oracle.topk_sample(y, k, 1.0, j / k)[2][0] == j

"""Pins of the oracle's temperature sampler (Gumbel-max over Philox4x64-10).

The generator is pinned to numpy's own Philox4x64-10 bit generator (a library
implementation of the same published definition); the Gumbel-max rule to what
it must produce mathematically: a draw from softmax(logits / T) (chi-square over
many counters), Gumbel(0, 1) noise (its mean and variance), the greedy argmax at
T <= 0, a near-uniform draw at a very large T, and NaN logits never drawn."""
import math

import numpy as np
import pytest

import oracle

scipy_stats = pytest.importorskip("scipy.stats")


def test_philox_matches_numpy_generator():
    rng = np.random.default_rng(7)
    for _ in range(20):
        ctr = rng.integers(1, 2 ** 63, size=4, dtype=np.uint64)
        key = rng.integers(0, 2 ** 63, size=2, dtype=np.uint64)
        # numpy's Philox increments the counter, then returns the block's four words
        bg = np.random.Philox(counter=np.array([ctr[0] - np.uint64(1), ctr[1], ctr[2], ctr[3]], np.uint64), key=key)
        want = [int(x) for x in bg.random_raw(4)]
        assert oracle.philox4x64_10([int(x) for x in ctr], [int(x) for x in key]) == want


def _draws(logits, T, n, seed=1234):
    return np.array([oracle.sample_f32(logits, T, seed, c) for c in range(n)])


def test_gumbel_max_draws_follow_softmax():
    logits = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4], np.float32)
    for T in (0.8, 3.0):
        d = _draws(logits, T, 40000)
        p = np.exp(logits.astype(np.float64) / T)
        p /= p.sum()
        obs = np.bincount(d, minlength=logits.size)
        stat, pval = scipy_stats.chisquare(obs, p * d.size)
        assert pval > 1e-4, (T, obs, p * d.size, pval)


def test_noise_is_standard_gumbel():
    g = np.array([oracle.gumbel_perturbed(0.0, v, 1.0, 99, 5) for v in range(60000)])
    assert abs(g.mean() - 0.5772156649) < 0.02
    assert abs(g.var() - math.pi ** 2 / 6) < 0.06
    # the noise is -log(-log u) with u in (0, 1): finite, and the largest values are rare
    assert np.all(np.isfinite(g))
    assert abs(np.mean(g > 2.0) - (1 - math.exp(-math.exp(-2.0)))) < 0.01


def test_temperature_zero_or_negative_is_greedy():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(1000).astype(np.float32)
    for T in (0.0, -1.0):
        assert oracle.sample_f32(x, T, 1, 2) == oracle.argmax_f32(x)


def test_very_high_temperature_is_near_uniform():
    logits = np.array([5.0, -5.0, 0.0, 2.0], np.float32)
    d = _draws(logits, 1e6, 20000, seed=8)
    obs = np.bincount(d, minlength=4)
    assert scipy_stats.chisquare(obs).pvalue > 1e-4


def test_draw_depends_on_seed_and_counter_only():
    x = np.random.default_rng(4).standard_normal(5000).astype(np.float32)
    a = [oracle.sample_f32(x, 1.0, 11, c) for c in range(50)]
    assert a == [oracle.sample_f32(x, 1.0, 11, c) for c in range(50)]  # deterministic
    assert len(set(a)) > 25  # different counters draw differently
    assert a != [oracle.sample_f32(x, 1.0, 12, c) for c in range(50)]


def test_nan_logits_are_never_drawn():
    x = np.array([np.nan, 0.0, np.nan, -1.0], np.float32)
    d = _draws(x, 2.0, 2000)
    assert set(d.tolist()) <= {1, 3}
    assert oracle.sample_f32(np.full(4, np.nan, np.float32), 1.0, 1, 1) == -1

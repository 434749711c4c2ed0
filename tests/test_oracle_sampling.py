"""Pins of the oracle's sampling head ("How Llama 3.1 Generates the Next Token",
Temperature, Softmax, Top-k and top-p sampling): the greedy limits, the draw
against the distribution it must realise (fraction of uniforms that pick each
token), the temperature's closed form, the pages' own top-k / top-p rules and a
brute-force smallest-set search for top-p."""
import itertools
import math

import numpy as np
import pytest

from oracle import sampling as sm

GRID = 20000
U = (np.arange(GRID) + 0.5) / GRID      # midpoints of a fine grid over [0, 1)


def _frequencies(z, temperature, top_k, top_p):
    ids = np.array([sm.sample_row(z, temperature, top_k, top_p, u) for u in U])
    return np.bincount(ids, minlength=len(z)) / GRID


def test_greedy_limits():
    rng = np.random.default_rng(0)
    z = rng.standard_normal(50)
    best = int(np.argmax(z))
    for u in (0.0, 0.3, 0.999):
        assert sm.sample_row(z, 0.0, 0, 1.0, u) == best           # T = 0
        assert sm.sample_row(z, 1.0, 1, 1.0, u) == best           # top_k = 1
        assert sm.sample_row(z, 1e-3, 0, 1.0, u) == best          # T -> 0 with a clear gap
    tie = np.array([0.5, 2.0, 2.0, -1.0])
    assert sm.sample_row(tie, 0.0, 0, 1.0, 0.7) == 1              # first maximum


def test_draw_realises_the_softmax():
    """No truncation: the share of uniforms choosing token i is P(i) = e^{z_i/T} / sum."""
    z = np.array([1.0, -0.5, 2.0, 0.25, 0.0, -3.0])
    for temperature in (1.0, 0.7, 1.8):
        want = np.exp(z / temperature) / np.sum(np.exp(z / temperature))
        assert np.allclose(_frequencies(z, temperature, 0, 1.0), want, atol=1.5 / GRID)


def test_temperature_closed_form():
    """softmax(z / T) = softmax(z)^(1/T) renormalised: T < 1 sharpens, T > 1 flattens."""
    rng = np.random.default_rng(1)
    z = rng.standard_normal(30) * 2
    p = sm.softmax_temperature(z, 1.0)
    for temperature in (0.5, 2.0):
        pt = sm.softmax_temperature(z, temperature)
        ref = p ** (1 / temperature)
        assert np.allclose(pt, ref / ref.sum(), rtol=1e-12)
    assert sm.softmax_temperature(z, 0.5).max() > p.max() > sm.softmax_temperature(z, 2.0).max()


def test_top_k_keeps_the_k_largest_renormalised():
    """[Next] Top-k: with top_k = 5 only the five most likely tokens are considered,
    renormalised to sum to one."""
    rng = np.random.default_rng(2)
    z = rng.standard_normal(40)
    freq = _frequencies(z, 1.0, 5, 1.0)
    top5 = np.argsort(-z)[:5]
    p = np.exp(z[top5]) / np.sum(np.exp(z[top5]))
    assert set(np.nonzero(freq)[0]) == set(top5)
    assert np.allclose(freq[top5], p, atol=1.5 / GRID)
    assert math.isclose(freq.sum(), 1.0)


def test_top_p_smallest_set_reaching_p():
    """[Next] Top-p: with top_p = 0.9, the most likely tokens are kept until their
    combined probability reaches or exceeds 90%."""
    assert sm.kept_count(np.array([0.5, 0.3, 0.15, 0.05]), 0, 0.9) == 3
    assert sm.kept_count(np.array([0.5, 0.4, 0.1]), 0, 0.9) == 2      # reaching it exactly is enough
    assert sm.kept_count(np.array([0.95, 0.04, 0.01]), 0, 0.9) == 1
    assert sm.kept_count(np.array([0.2] * 5), 0, 1.0) == 5


@pytest.mark.parametrize("seed", range(6))
def test_top_p_matches_brute_force_subsets(seed):
    rng = np.random.default_rng(10 + seed)
    V = 7
    z = rng.standard_normal(V) * 1.5
    p = sm.softmax_temperature(z, 1.0)
    top_p = float(rng.uniform(0.3, 0.99))
    # the smallest subset of any tokens whose mass is at least top_p
    smallest = min(len(s) for r in range(1, V + 1) for s in itertools.combinations(range(V), r)
                   if p[list(s)].sum() >= top_p)
    n = sm.kept_count(p[sm.descending_order(z)], 0, top_p)
    assert n == smallest
    freq = _frequencies(z, 1.0, 0, top_p)
    kept = sm.descending_order(z)[:n]
    assert set(np.nonzero(freq)[0]) == set(kept)
    assert np.allclose(freq[kept], p[kept] / p[kept].sum(), atol=1.5 / GRID)


def test_top_k_and_top_p_together_keep_the_shorter_prefix():
    p = np.array([0.4, 0.3, 0.2, 0.06, 0.04])
    assert sm.kept_count(p, 2, 0.95) == 2       # top-k is the tighter restriction
    assert sm.kept_count(p, 4, 0.6) == 2        # top-p is the tighter one
    assert sm.kept_count(p, 0, 0.95) == 4


def test_equal_logits_are_drawn_in_index_order():
    z = np.array([0.0, 1.0, 1.0, 1.0])
    freq = _frequencies(z, 1.0, 3, 1.0)
    assert np.allclose(freq, [0, 1 / 3, 1 / 3, 1 / 3], atol=1.5 / GRID)
    assert sm.sample_row(z, 1.0, 3, 1.0, 0.1) == 1 and sm.sample_row(z, 1.0, 3, 1.0, 0.9) == 3
    # a tie cut by top-k keeps the lower indices
    freq = _frequencies(z, 1.0, 2, 1.0)
    assert np.allclose(freq, [0, 0.5, 0.5, 0], atol=1.5 / GRID)

"""Pins for oracle/philox.py: published Philox known answers and the Gumbel-max law."""
import numpy as np
import pytest

from conftest import golden_lines
from oracle.philox import gumbel_row, philox4x32_10, uniform_open01


def test_philox4x32_10_known_answers():
    rows = golden_lines("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        w = [int(x, 16) for x in r]
        out = philox4x32_10(w[0:4], w[4:6])
        assert [int(o) for o in out] == w[6:10]


def test_philox_vectorised_matches_scalar():
    ctr = np.arange(17, dtype=np.uint64)
    vec = philox4x32_10((ctr, 5, 9, 11), (123, 456))
    for j in range(17):
        sc = philox4x32_10((j, 5, 9, 11), (123, 456))
        assert [int(v[j]) for v in vec] == [int(s) for s in sc]


def test_uniform_is_open_and_exact_in_fp32():
    x = np.array([0, 1, 511, 512, 0xFFFFFFFF, 0x80000000], dtype=np.uint32)
    u = uniform_open01(x)
    assert np.all(u > 0) and np.all(u < 1)
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert u[0] == 2.0 ** -24 and u[4] == 1 - 2.0 ** -24


def test_gumbel_rows_are_keyed_by_position_and_sequence():
    a = gumbel_row(7, 0, 100, 1000)
    assert np.array_equal(a, gumbel_row(7, 0, 100, 1000))
    assert not np.array_equal(a, gumbel_row(7, 0, 101, 1000))
    assert not np.array_equal(a, gumbel_row(7, 1, 100, 1000))
    assert not np.array_equal(a, gumbel_row(8, 0, 100, 1000))
    # a longer row extends a shorter one
    assert np.array_equal(gumbel_row(7, 0, 100, 1003)[:1000], a)


def test_gumbel_moments():
    g = gumbel_row(11, 0, 3, 400000)
    assert g.mean() == pytest.approx(np.euler_gamma, abs=0.01)
    assert g.var() == pytest.approx(np.pi ** 2 / 6, abs=0.03)


def test_gumbel_max_samples_softmax():
    """Gumbel-max trick: argmax(l / tau + G) ~ softmax(l / tau) (chi-square test)."""
    from scipy.stats import chisquare
    V, tau, n = 8, 0.7, 100000
    logits = np.array([0.3, -1.0, 1.2, 0.0, 0.9, -0.4, 0.5, 1.1])
    counts = np.zeros(V)
    for pos in range(n):
        g = gumbel_row(2, 0, pos, V)
        counts[np.argmax(logits / tau + g)] += 1
    p = np.exp(logits / tau)
    p /= p.sum()
    stat, pval = chisquare(counts, p * n)
    assert pval > 1e-3, (counts, p * n)

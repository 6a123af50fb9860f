"""Pins for oracle/analysis.py: the paper's worked examples, closed forms and invariants."""
import random

import pytest

from conftest import golden_lines
from oracle import analysis as A


def _golden(name):
    return {ln[0]: [int(x) for x in ln[1:]] for ln in golden_lines(name)}


def test_appendix_a3_worked_example():
    g = _golden("appendix_a3_exploration_example.txt")
    L, X, e = g["L"][0], g["X"], g["ead"][0]
    assert A.depth_ceiling(e, X) == g["depth_ceiling"][0]
    assert A.exploration_workload(e, X) == g["depth_ceiling"][0]
    assert A.exploration_overhead(e, X) == g["overhead"][0]
    assert A.resolution(X, L) == g["resolution"][0]


def test_appendix_a2_worked_example():
    g = _golden("appendix_a2_selection_example.txt")
    L, e = g["L"][0], g["ead"][0]
    s_ok = g["accepted_selection"][0]
    assert A.selection_overhead(1.0, [s_ok], L, e) == g["accepted_overhead"][0]
    assert A.selection_workload(1.0, [s_ok], L) == s_ok
    s_bad = g["failed_selection"][0]
    for s1, s2 in [(4, 4), (7, 11), (1, 19)]:
        W = A.selection_workload(0.0, [s_bad, s1, s2], L)
        assert W - s1 - s2 == g["failed_constant"][0]
        assert W > L or s1 + s2 <= -4      # "can exceed the 20-layer cost of AR"


@pytest.mark.parametrize("X,L,delta", [
    ([2, 4, 6, 8], 8, 1), ([8, 16, 24, 32], 32, 7), (list(range(4, 33, 4)), 32, 3),
    ([9, 18, 27, 36], 36, 8), ([36], 36, 35), (list(range(1, 33)), 32, 0)])
def test_resolution_of_workload_sets(X, L, delta):
    assert A.resolution(X, L) == delta


def test_resolution_uniform_is_spacing_minus_one():
    for L in (8, 20, 32, 36, 48, 80):
        for K in range(1, 9):
            if L % K == 0:
                assert A.resolution(A.uniform_exploration_set(L, K), L) == L // K - 1


def test_ead_definitions_brute_force():
    rng = random.Random(0)
    for _ in range(500):
        L = rng.randint(1, 12)
        omega = [rng.randint(0, 1) for _ in range(L - 1)] + [1]
        e = A.ead(omega)
        assert omega[e - 1] == 1 and all(o == 0 for o in omega[:e - 1])
        es = A.ead_stable(omega)
        assert all(omega[n - 1] == 1 for n in range(es, L + 1))
        assert es == 1 or omega[es - 2] == 0
        assert e <= es


def test_prop6_overhead_bounded_by_resolution():
    rng = random.Random(1)
    for _ in range(300):
        L = rng.randint(2, 40)
        X = sorted(set(rng.sample(range(1, L), rng.randint(0, L - 2))) | {L})
        d = A.resolution(X, L)
        for e in range(1, L + 1):
            c = A.exploration_overhead(e, X)
            assert 0 <= c <= d
        # the maximum is attained (Delta is the largest rounding error)
        assert max(A.exploration_overhead(e, X) for e in range(1, L + 1)) == d


def test_eq8_equals_eq9():
    rng = random.Random(2)
    for _ in range(300):
        L = rng.randint(2, 20)
        X = sorted(set(rng.sample(range(1, L), rng.randint(0, L - 2))) | {L})
        omega = [rng.randint(0, 1) for _ in range(L - 1)] + [1]
        assert A.exploration_workload_from_omega(omega, X) == A.exploration_workload(A.ead_stable(omega), X)


def test_eq14_bounds_and_monotonicity():
    rng = random.Random(3)
    for _ in range(200):
        L = rng.randint(2, 40)
        T = rng.randint(1, 30)
        eads = [rng.randint(1, L) for _ in range(T)]
        X = sorted(set(rng.sample(range(1, L), rng.randint(0, L - 2))) | {L})
        lo, sx, se = A.exploration_speedup_bounds(eads, X, L)
        assert 1.0 <= lo + 1e-12 and lo <= sx + 1e-12 and sx <= se + 1e-12
        assert sx == pytest.approx(A.speedup([A.depth_ceiling(e, X) for e in eads], L))
        Xp = sorted(set(X) | set(rng.sample(range(1, L + 1), rng.randint(0, L))))
        _, sxp, _ = A.exploration_speedup_bounds(eads, Xp, L)
        assert sx <= sxp + 1e-12 <= se + 2e-12
        # X = [L] reaches the EAD oracle
        _, sfull, _ = A.exploration_speedup_bounds(eads, list(range(1, L + 1)), L)
        assert sfull == pytest.approx(se)


def test_speedup_of_ar_is_one():
    assert A.speedup([32] * 10, 32) == 1.0
    assert A.speedup([8, 16], 32) == pytest.approx(64 / 24)

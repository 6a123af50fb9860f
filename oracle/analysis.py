"""Depth-readiness quantities of "Depth Exploration for LLM Decoding", section 2.

Each function restates one definition or equation of the paper (arXiv 2606.29223):
acceptance and (stable) earliest available depth (Def. 1, Eq. 1-3), depth selection
cost (Def. 2, Eq. 4; Prop. 3, Eq. 5), the exploration set, depth ceiling and
resolution (Def. 4, Eq. 6-7), the exploration workload and its overhead (Def. 5,
Eq. 8-11; Prop. 6) and the depth-side speedup with its bounds (Prop. 7, Eq. 12-14).
Depths are 1-based layer counts in [L] = {1, ..., L}.
"""
from __future__ import annotations

from typing import Sequence


def ead(omega: Sequence[int]) -> int:
    """Eq. 1: EAD(t) = min{l in [L] : Omega(t, l) = 1}; omega[l-1] = Omega(t, l), Omega(t, L) = 1."""
    L = len(omega)
    assert omega[L - 1] == 1, "Omega(t, L) = 1 by construction (Def. 1)"
    for l in range(1, L + 1):
        if omega[l - 1]:
            return l
    raise AssertionError("unreachable")


def stable_acceptance(omega: Sequence[int]):
    """Eq. 2: Omega^stab(t, l) = 1 iff Omega(t, n) = 1 for all n in {l, ..., L}."""
    L = len(omega)
    out = [0] * L
    ok = 1
    for l in range(L, 0, -1):
        ok = ok and omega[l - 1]
        out[l - 1] = 1 if ok else 0
    return out


def ead_stable(omega: Sequence[int]) -> int:
    """Eq. 3: the stable earliest available depth."""
    return ead(stable_acceptance(omega))


def depth_ceiling(l: int, X: Sequence[int]) -> int:
    """Eq. 6: ceil(l)_X = min{d in X : d >= l}."""
    return min(d for d in X if d >= l)


def resolution(X: Sequence[int], L: int) -> int:
    """Eq. 7: Delta(X) = max over l in [L] of (ceil(l)_X - l)."""
    assert max(X) == L, "the final depth is always explored (Def. 4)"
    return max(depth_ceiling(l, X) - l for l in range(1, L + 1))


def exploration_workload(ead_t: int, X: Sequence[int]) -> int:
    """Eq. 9: W_X(t) = ceil(EAD(t))_X (equivalently Eq. 8 under stable readiness)."""
    return depth_ceiling(ead_t, X)


def exploration_workload_from_omega(omega: Sequence[int], X: Sequence[int]) -> int:
    """Eq. 8: W_X(t) = min{d in X : Omega^stab(t, d) = 1}."""
    stab = stable_acceptance(omega)
    return min(d for d in X if stab[d - 1])


def exploration_overhead(ead_t: int, X: Sequence[int]) -> int:
    """Eq. 10: c^exp_t = ceil(EAD(t))_X - EAD(t)."""
    return depth_ceiling(ead_t, X) - ead_t


def selection_workload(p_acc: float, s: Sequence[int], L: int) -> float:
    """Eq. 4: W^sel_t = p s_t + (1 - p) (L + sum_{i=t}^{t+v_t-1} s_i); s = [s_t, ..., s_{t+v_t-1}]."""
    return p_acc * s[0] + (1.0 - p_acc) * (L + sum(s))


def selection_overhead(p_acc: float, s: Sequence[int], L: int, ead_t: int) -> float:
    """Eq. 5: c^sel_t = p (s_t - EAD) + (1 - p)(L + sum s_i - EAD)."""
    return p_acc * (s[0] - ead_t) + (1.0 - p_acc) * (L + sum(s) - ead_t)


def speedup(W: Sequence[float], L: int) -> float:
    """Eq. 12: S = L T / sum_t W(t)."""
    return L * len(W) / float(sum(W))


def exploration_speedup_bounds(eads: Sequence[int], X: Sequence[int], L: int):
    """Eq. 13-14: (lower bound, S_X, S_EAD) with 1 <= lower <= S_X <= S_EAD."""
    T = len(eads)
    delta = resolution(X, L)
    lower = L * T / float(sum(min(e + delta, L) for e in eads))
    s_x = L * T / float(sum(depth_ceiling(e, X) for e in eads))
    s_ead = L * T / float(sum(eads))
    return lower, s_x, s_ead


def uniform_exploration_set(L: int, K: int):
    """DEX-1/K: K explorers, each covering L/K layers (section 4 setup); requires K | L."""
    assert L % K == 0
    return [L // K * (k + 1) for k in range(K)]

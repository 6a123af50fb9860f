"""Pins for the decision helpers of oracle/dex.py that every GPU parity test leans on.

``margin`` (top-1 minus top-2 of the finite decision scores) decides which tokens the
parity tests compare, and ``first_argmax`` is the tie rule of every decode.  The values
below are worked by hand; the sampled cases pin properties that fail if the margin were
taken on the raw logits or without the temperature ("Depth Exploration for LLM
Decoding", Appendix C.1: the decision is argmax of logits / tau + Gumbel noise in
sampling mode, argmax of the logits in greedy mode; section 3.3: DECS excludes the
shallower proposals of the slot chain, except at the final-depth reference).
"""
import math

import numpy as np
import pytest

from oracle import dex


def test_margin_of_a_known_gap():
    assert dex.margin(np.array([0.0, 2.5, 1.0, 2.25])) == 0.25
    assert dex.margin(np.array([-3.0, -1.0])) == 2.0
    assert dex.first_argmax(np.array([0.0, 2.5, 1.0, 2.25])) == 1


def test_margin_ignores_masked_entries():
    inf = math.inf
    # the masked -inf entries are neither top-1 nor top-2
    assert dex.margin(np.array([-inf, 3.0, -inf, 1.0])) == 2.0
    # one finite score left: no runner-up, the decision cannot flip
    assert dex.margin(np.array([-inf, 0.5, -inf])) == inf
    assert dex.first_argmax(np.array([-inf, -inf, 2.0, 2.0])) == 2


def test_tie_has_zero_margin_and_lowest_id():
    s = np.array([1.0, 4.0, 4.0, 2.0])
    assert dex.margin(s) == 0.0
    assert dex.first_argmax(s) == 1
    assert dex.first_argmax(np.array([7.0, 1.0, 7.0])) == 0


def test_exclusion_moves_the_token_and_the_margin():
    """Excluding the top token of a non-final depth: the decision falls to the runner-up and
    the margin is taken between the 2nd and 3rd logits; the final depth ignores the
    exclusion."""
    z = np.array([0.5, 3.0, 2.0, 1.25, -1.0])
    tok, mg, excl = dex.depth_coupled_token(z, [1], False, dex.Rule(), 0, 10)
    assert (tok, mg, excl) == (2, 0.75, [1])
    tok, mg, excl = dex.depth_coupled_token(z, [1], True, dex.Rule(), 0, 10)
    assert (tok, mg, excl) == (1, 1.0, [])
    tok, mg, excl = dex.depth_coupled_token(z, [1, 2, 1], False, dex.Rule(), 0, 10)
    assert (tok, mg, excl) == (3, 0.75, [1, 2])
    # decoding without DECS: nothing excluded
    tok, mg, excl = dex.depth_coupled_token(z, [1], False, dex.Rule(), 0, 10, enabled=False)
    assert (tok, mg, excl) == (1, 1.0, [])


@pytest.mark.parametrize("seed,pos", [(5, 7), (11, 300)])
def test_sampled_margin_is_taken_on_the_noisy_scores(seed, pos):
    V = 64
    rule = dex.Rule(sample=True, tau=0.5, seed=seed)
    flat = np.zeros(V)
    # raw logits all equal: a margin on the logits would be 0, on l / tau + G it is not
    assert dex.margin(dex.decision_scores(flat, dex.Rule(), 0, pos)) == 0.0
    m_flat = dex.margin(dex.decision_scores(flat, rule, 0, pos))
    assert m_flat > 0.0
    # a constant shift of the logits moves every score alike: same margin
    assert dex.margin(dex.decision_scores(flat + 3.0, rule, 0, pos)) == pytest.approx(m_flat, abs=1e-12)
    # the temperature divides the logits: logits 2x at tau = 0.5 decide like x at tau = 1
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(V)
    a = dex.margin(dex.decision_scores(x / 2.0, rule, 0, pos))
    b = dex.margin(dex.decision_scores(x / 4.0, dex.Rule(sample=True, tau=0.25, seed=seed), 0, pos))
    c = dex.margin(dex.decision_scores(x, dex.Rule(sample=True, tau=1.0, seed=seed), 0, pos))
    assert a == pytest.approx(c, abs=1e-12) and b == pytest.approx(c, abs=1e-12)
    # and it is not the logits' own margin
    assert c != pytest.approx(dex.margin(x), abs=1e-9)


def test_sampled_exclusion_keeps_masked_ids_out_of_the_margin():
    """A masked id gets -inf before the noise is added, so it can never be the top-1 or the
    top-2 of the sampled scores, however large its logit."""
    V = 32
    rule = dex.Rule(sample=True, tau=0.7, seed=3)
    z = np.zeros(V)
    z[4] = 100.0
    tok, mg, excl = dex.depth_coupled_token(z, [4], False, rule, 0, 9)
    assert tok != 4 and excl == [4]
    ref = dex.decision_scores(np.where(np.arange(V) == 4, -np.inf, z), rule, 0, 9)
    assert mg == dex.margin(ref) and np.isfinite(mg)
    # unmasked, the id with logit 100 wins by far more than any Gumbel gap
    tok, mg, _ = dex.depth_coupled_token(z, [4], True, rule, 0, 9)
    assert tok == 4 and mg > 100.0 / 0.7 - 40.0

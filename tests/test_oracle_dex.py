"""Pins for Algorithm 1 / Algorithm 2 in oracle/dex.py on tiny models.

What the paper fixes: DEX commits exactly the AR stream (section 3.2, lossless
invariant); the committed token is the unmasked final-depth token (section 3.3,
Appendix C.1); commit selects the shallowest matching anchor branch (section 3.2);
the per-token charge relates to EAD as in Def. 1-5 / Prop. 6.
"""
import numpy as np
import pytest

from conftest import tiny_model
from oracle import analysis as A
from oracle import dex

import dex_inputs as di

PROMPT = di.gen_prompts(di.TINY, 1, 32)[0].tolist()
VARIANTS = [(0.1, True), (0.3, False), (1.0, False)]


def _run(alpha, tied, X, T, rule, use_decs=True, prompt=PROMPT, n_layers=8):
    _, _, m = tiny_model(alpha, tied, n_layers)
    ar = dex.ar_generate(m, prompt, T, rule=rule, record_depths=True)
    r = dex.dex_generate(m, prompt, X, T, rule=rule, use_decs=use_decs)
    return m, ar, r


@pytest.mark.parametrize("alpha,tied", VARIANTS)
@pytest.mark.parametrize("X", [[2, 4, 6, 8], [4, 8], [1, 2, 3, 4, 5, 6, 7, 8], [8], [1, 8]])
@pytest.mark.parametrize("sample", [False, True])
def test_dex_is_lossless(alpha, tied, X, sample):
    rule = dex.Rule(sample=sample, tau=0.7, seed=2)
    m, ar, r = _run(alpha, tied, X, 12, rule)
    assert r.tokens == ar.tokens
    N = len(X)
    for c, y in zip(r.commits, ar.tokens):
        assert c.token == y
    # the final-depth reference is never masked; only the anchor reaches stage N-1
    for nd in r.nodes:
        if nd.stage == N - 1:
            assert nd.node == dex.anchor_node(N - 1) and nd.masked == []


def test_dex_lossless_without_decs_and_other_prompts():
    for seed in (3, 4):
        prompt = di.uniform_ids(9, 4096, seed, 99).tolist()
        for use_decs in (False, True):
            _, ar, r = _run(1.0, False, [2, 4, 6, 8], 10, dex.Rule(), use_decs, prompt)
            assert r.tokens == ar.tokens


@pytest.mark.parametrize("sample", [False, True])
def test_ead_and_charge_relations(sample):
    """c14: (1) vanilla greedy k* is the first explored depth whose candidate is y;
    (2) d_{k*} <= ceil(EAD^stab)_X always; (3) equality without non-stable early hits;
    (4) 0 <= W_X - EAD^stab <= Delta(X)."""
    rule = dex.Rule(sample=sample, tau=0.7, seed=5)
    for alpha, tied in VARIANTS[1:]:
        X = [2, 4, 6, 8]
        L = 8
        m, ar, vanilla = _run(alpha, tied, X, 16, rule, use_decs=False)
        decs = dex.dex_generate(m, PROMPT, X, 16, rule=rule, use_decs=True)
        omegas, eads, stabs = dex.ead_profile(ar)
        dv, dd = vanilla.depth_charges(X), decs.depth_charges(X)
        for t in range(16):
            first_hit = min(d for d in X if omegas[t][d - 1])
            assert dv[t] == first_hit                                         # (1)
            W = A.exploration_workload(stabs[t], X)
            assert dd[t] <= dv[t] <= W                                        # (2) and DECS never later
            if not any(omegas[t][d - 1] for d in X if d < W):
                assert dv[t] == W                                             # (3)
            assert 0 <= W - stabs[t] <= A.resolution(X, L)                   # (4)
            assert eads[t] <= stabs[t]


def test_decs_diversifies_slot_chains():
    _, _, m = tiny_model(1.0, False)
    r = dex.dex_generate(m, PROMPT, [1, 2, 3, 4, 5, 6, 7, 8], 8, use_decs=True)
    N = 8
    by_round = {}
    for nd in r.nodes:
        by_round.setdefault(nd.round, {})[nd.node] = nd
    checked = 0
    for rnd, nodes in by_round.items():
        for i, nd in nodes.items():
            if nd.stage == N - 1:
                continue
            # masked set = tokens of the shallower members of the slot chain, and the
            # decoded token avoids them
            assert nd.token not in nd.masked
            assert len(nd.masked) <= nd.stage
            checked += len(nd.masked)
    assert checked > 0


def test_final_token_equals_unmasked_gumbel_max():
    rule = dex.Rule(sample=True, tau=0.7, seed=9)
    _, _, m = tiny_model(1.0, False)
    r = dex.dex_generate(m, PROMPT, [2, 4, 6, 8], 6, rule=rule, keep_logits=True)
    n_ref = 0
    for nd in r.nodes:
        if nd.stage == 3:
            score = nd.logits / rule.tau + dex.gumbel_row(rule.seed, 0, nd.target_pos, nd.logits.size)
            assert nd.token == int(np.argmax(score))
            n_ref += 1
    assert n_ref == 6


def test_rounds_per_commit_and_layer_accounting():
    X = [2, 4, 6, 8]
    N = len(X)
    _, _, m = tiny_model(0.3, False)
    r = dex.dex_generate(m, PROMPT, X, 20)
    assert r.commits[0].rounds == N                      # first cycle starts from q = 0
    for prev, cur in zip(r.commits, r.commits[1:]):
        assert cur.rounds == prev.kstar + 1              # q' = N - k* - 1
    assert r.rounds == sum(c.rounds for c in r.commits)
    per_round_nodes = {}
    for nd in r.nodes:
        per_round_nodes.setdefault(nd.round, []).append(nd)
    passes, node_layers = 0, 0
    for rnd, nodes in per_round_nodes.items():
        q = nodes[0].q
        assert len(nodes) == 2 ** q
        passes += X[q]                                   # a round at state q streams layers 1..d_q
        node_layers += sum(X[n.stage] - (X[n.stage - 1] if n.stage else 0) for n in nodes)
    assert r.layer_passes == passes and r.node_layers == node_layers


def test_degenerate_tiny_repeats_last_token():
    """alpha = 0.1 with the tied head: the input token's own logit dominates, so greedy
    repeats the last prompt token and every commit hits at the shallowest depth."""
    _, ar, r = _run(0.1, True, [2, 4, 6, 8], 12, dex.Rule())
    assert set(ar.tokens) == {PROMPT[-1]}
    assert all(c.kstar == 0 for c in r.commits)


# ---- sparse lattice (speculation cap) -------------------------------------------------------

@pytest.mark.parametrize("X", [[2, 4, 6, 8], [1, 2, 3, 4, 5, 6, 7, 8]])
@pytest.mark.parametrize("cap", [1, 2, 3])
def test_sparse_lattice_is_lossless(X, cap):
    """Pruned branches never carry the commit: the stream equals plain AR for any cap."""
    shape, w, m = tiny_model(alpha=1.0, tied=False)
    prompt = di.gen_prompts(shape, 1, 16)[0].tolist()
    ar = dex.ar_generate(m, prompt, 12)
    r = dex.dex_generate(m, prompt, X, 12, max_branch=cap)
    assert r.tokens == ar.tokens
    for nd in r.nodes:   # every node respects the cap
        assert nd.plen <= cap


def test_sparse_lattice_with_cap_at_least_n_minus_1_is_the_full_lattice():
    """plen <= q <= N-1 always, so a cap of N-1 prunes nothing: same nodes, same rounds."""
    shape, w, m = tiny_model(alpha=0.3, tied=False)
    prompt = di.gen_prompts(shape, 1, 16)[0].tolist()
    X = [2, 4, 6, 8]
    full = dex.dex_generate(m, prompt, X, 10)
    capped = dex.dex_generate(m, prompt, X, 10, max_branch=len(X) - 1)
    assert full.tokens == capped.tokens and full.rounds == capped.rounds
    assert [(n.round, n.node, n.token) for n in full.nodes] == [(n.round, n.node, n.token) for n in capped.nodes]


@pytest.mark.parametrize("cap", [1, 2])
def test_sparse_lattice_first_cycle_counts(cap):
    """Before the first commit the lattice is fresh: the level-q round holds the paths of q
    moves with at most `cap` position moves, sum_{p <= cap} C(q, p) nodes (counted here by
    brute force over move strings)."""
    from itertools import product
    shape, w, m = tiny_model(alpha=0.3, tied=False)
    prompt = di.gen_prompts(shape, 1, 16)[0].tolist()
    X = [1, 2, 3, 4, 5, 6, 7, 8]
    r = dex.dex_generate(m, prompt, X, 1, max_branch=cap)
    per_round = {}
    for nd in r.nodes:
        per_round[nd.round] = per_round.get(nd.round, 0) + 1
    for q in range(len(X)):
        brute = sum(1 for moves in product("DP", repeat=q) if moves.count("P") <= cap)
        assert per_round[q] == brute, (q, per_round[q], brute)


# ---- inducing adapters (Appendix C.2) --------------------------------------------------------

def _adapter(rng, d, alpha, zero_w2=False):
    ad = {"g": 1.0 + 0.1 * rng.standard_normal(d), "w1": 0.1 * rng.standard_normal((2 * d, d)),
          "b1": 0.1 * rng.standard_normal(2 * d), "w2": 0.1 * rng.standard_normal((d, 2 * d)),
          "b2": 0.1 * rng.standard_normal(d), "alpha": alpha}
    if zero_w2:
        ad["w2"] = np.zeros((d, 2 * d))
    return ad


def test_adapter_special_cases():
    from oracle.model import apply_adapter
    from scipy.special import expit
    rng = np.random.default_rng(0)
    d = 16
    h = rng.standard_normal((3, d))
    # alpha = 0: the plain hidden state
    assert np.array_equal(apply_adapter(h, _adapter(rng, d, 0.0), 1e-5), h)
    # W2 = 0: h + alpha b2 whatever W1, b1, g
    ad = _adapter(rng, d, 0.7, zero_w2=True)
    assert np.allclose(apply_adapter(h, ad, 1e-5), h + 0.7 * ad["b2"], rtol=0, atol=1e-15)
    # W1 = [I; 0], b1 = 0, W2 = [I, 0]: h + alpha (SiLU(RMSNorm(h; g)) + b2), SiLU = x expit(x)
    ad = _adapter(rng, d, 0.5)
    ad["w1"] = np.vstack([np.eye(d), np.zeros((d, d))])
    ad["b1"] = np.zeros(2 * d)
    ad["w2"] = np.hstack([np.eye(d), np.zeros((d, d))])
    n = h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + 1e-5) * ad["g"]
    assert np.allclose(apply_adapter(h, ad, 1e-5), h + 0.5 * (n * expit(n) + ad["b2"]), rtol=1e-13, atol=1e-13)


def test_adapter_correction_is_scale_invariant():
    """The correction depends on h only through RMSNorm(h): with eps = 0, scaling h by a
    positive factor leaves h~ - h unchanged."""
    from oracle.model import apply_adapter
    rng = np.random.default_rng(1)
    d = 32
    h = rng.standard_normal((2, d))
    ad = _adapter(rng, d, 0.4)
    d1 = apply_adapter(h, ad, 0.0) - h
    d2 = apply_adapter(7.5 * h, ad, 0.0) - 7.5 * h
    assert np.allclose(d1, d2, rtol=1e-12, atol=1e-12)


def _widened_adapters(shape, X, gate):
    from oracle.model import widen_bf16
    ads = di.gen_adapters(shape, X, gate=gate)
    return [{k: (v if k == "alpha" else widen_bf16(di.bf16_bits(v))) for k, v in a.items()} for a in ads]


@pytest.mark.parametrize("sample", [False, True])
def test_adapters_keep_dex_lossless_and_change_proposals(sample):
    shape, w, m = tiny_model(alpha=0.3, tied=False)
    prompt = di.gen_prompts(shape, 1, 16)[0].tolist()
    X = [2, 4, 6, 8]
    rule = dex.Rule(sample=sample, tau=0.7, seed=3)
    ads = _widened_adapters(shape, X, gate=2.0)
    ar = dex.ar_generate(m, prompt, 12, rule=rule)
    plain = dex.dex_generate(m, prompt, X, 12, rule=rule)
    adapted = dex.dex_generate(m, prompt, X, 12, rule=rule, adapters=ads)
    assert adapted.tokens == ar.tokens == plain.tokens
    # in the first cycle (before any commit) both lattices hold the same prefixes: the
    # final-depth node is never adapted, intermediate proposals are
    first = {(n.round, n.node): n for n in plain.nodes if n.round < len(X)}
    changed = 0
    for n in adapted.nodes:
        if n.round >= len(X):
            continue
        o = first[(n.round, n.node)]
        if n.stage == len(X) - 1:
            assert n.token == o.token
        elif n.token != o.token:
            changed += 1
    assert changed > 0


def test_decoding_from_a_prefilled_cache_is_the_same_decode():
    """A prefilled cache reused across decodes (the benchmark's CPU leg) gives the same
    tokens, logits and nodes as prefilling inside each call, any number of times."""
    shape, w, m = tiny_model(alpha=0.3, tied=False)
    prompt = di.gen_prompts(shape, 1, 16)[0].tolist()
    X = [2, 4, 6, 8]
    T = 6
    plain = dex.dex_generate(m, prompt, X, T, keep_logits=True)
    cache = dex.prefill(m, prompt, len(prompt) + T + len(X) + 1)
    for _ in range(2):
        again = dex.dex_generate(m, prompt, X, T, keep_logits=True, cache=cache)
        assert again.tokens == plain.tokens and again.rounds == plain.rounds
        for a, b in zip(again.nodes, plain.nodes):
            assert (a.node, a.token) == (b.node, b.token) and np.array_equal(a.logits, b.logits)
    ar = dex.ar_generate(m, prompt, T, cache=cache)
    assert ar.tokens == dex.ar_generate(m, prompt, T).tokens == plain.tokens

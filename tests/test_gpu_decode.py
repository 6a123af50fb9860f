"""End-to-end GPU parity of DEX rounds.

* the DEX token stream equals the library's own AR stream, bit for bit, and so do the
  final-depth logits of every committed token (the lossless invariant of section 3.2,
  checked on one GPU with row-wise arithmetic that does not depend on the batch);
* AR logits are within 5e-2 of the fp64 oracle and tokens equal the oracle's wherever
  its top-1/top-2 margin exceeds 0.1;
* every lattice node's token equals the oracle's Algorithm 1 node where margins allow;
* batch invariance: a sequence decodes identically alone and inside a batch.
"""
import numpy as np
import pytest

import dex_inputs as di
from gpu_util import check_logits_and_tokens, oracle_model, require_gpu
from oracle import dex as odex

pytestmark = pytest.mark.gpu

SMALL = di.ModelShape(n_layers=4, d_model=1024, n_heads=8, n_kv_heads=8, head_dim=128, d_ff=2816,
                      vocab=8192, tied_head=False)
SMALL_GQA = di.ModelShape(n_layers=4, d_model=1024, n_heads=16, n_kv_heads=4, head_dim=64, d_ff=2816,
                          vocab=8192, tied_head=False, rope_theta=1e6)
# sixteen query heads per KV head: a node row alone exceeds one attention pass (8 queries),
# so decode items take the multi-pass attention variant
SMALL_GQA16 = di.ModelShape(n_layers=4, d_model=2048, n_heads=16, n_kv_heads=1, head_dim=128, d_ff=5632,
                            vocab=8192, tied_head=False, rope_theta=1e6)
TINY_UNTIED = di.ModelShape(**{**di.TINY.__dict__, "tied_head": False})


def _ar_with_logits(dec, T):
    ys, zs = [], []
    for _ in range(T):
        tok, nc = dec.step(ar=True)
        assert nc[0] == 1
        ys.append(tok[0])
        zs.append(dec.debug_logits()[0].copy())
    return ys, zs


def _dex_with_final_logits(dec, N, T):
    """Run DEX rounds; return committed tokens and the logits of each final-depth node."""
    ys, zs = [], []
    while len(ys) < T:
        tok, nc = dec.step()
        nodes = dec.last_round_nodes()
        if nc[0]:
            ys.append(tok[0])
            lg = dec.debug_logits()
            k = [i for i, nd in enumerate(nodes) if nd["stage"] == N - 1]
            assert len(k) == 1
            zs.append(lg[k[0]].copy())
    return ys, zs


CASES = [
    ("tiny", di.TINY, 0.1, [2, 4, 6, 8], 24),
    ("tiny_untied_a03", TINY_UNTIED, 0.3, [2, 4, 6, 8], 24),
    ("tiny_untied_a1_x8", TINY_UNTIED, 1.0, [1, 2, 3, 4, 5, 6, 7, 8], 16),
    ("small_split_k", SMALL, 0.3, [1, 2, 3, 4], 16),
    ("small_gqa_hd64", SMALL_GQA, 0.3, [2, 4], 16),
    ("small_gqa16", SMALL_GQA16, 0.3, [2, 4], 16),
]


@pytest.mark.parametrize("name,shape,alpha,X,T", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("sample", [False, True])
def test_dex_equals_ar_and_oracle(name, shape, alpha, X, T, sample):
    dexlib = require_gpu()
    w = di.gen_weights(shape, alpha, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 40)[0].tolist()   # 39 prefilled positions: a ragged key group
    dec = dexlib.Decoder(shape, w, X, batch=1, max_ctx=256, max_new=T, sample=sample, tau=0.7, seed=11,
                         debug_logits=True)
    try:
        dec.prefill(0, prompt)
        y_dex, z_dex = _dex_with_final_logits(dec, len(X), T)
        st = dec.stats()
        dec.prefill(0, prompt)
        y_ar, z_ar = _ar_with_logits(dec, T)
    finally:
        dec.close()
    assert y_dex == y_ar
    for t in range(T):
        assert np.array_equal(z_dex[t].view(np.uint32), z_ar[t].view(np.uint32)), f"token {t}: logits differ"
    assert st["commits"] == T
    m = oracle_model(shape, w)
    rule = odex.Rule(sample=sample, tau=0.7, seed=11)
    ref = odex.ar_generate(m, prompt, T, rule=rule, force=y_ar)
    scores = [odex.decision_scores(ref.logits[t], rule, 0, len(prompt) + t) for t in range(T)]
    check_logits_and_tokens(z_ar, y_ar, ref, scores=scores)


def test_lattice_nodes_match_oracle_algorithm1():
    dexlib = require_gpu()
    shape, X, T = TINY_UNTIED, [2, 4, 6, 8], 16
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 32)[0].tolist()
    dec = dexlib.Decoder(shape, w, X, batch=1, max_ctx=128, max_new=T, debug_logits=True)
    m = oracle_model(shape, w)
    ref = odex.dex_generate(m, prompt, X, T, keep_logits=True)
    rounds = {}
    for nd in ref.nodes:
        rounds.setdefault(nd.round, {})[nd.node] = nd
    try:
        dec.prefill(0, prompt)
        checked, worst = 0, 0.0
        for r in range(ref.rounds):
            dec.step()
            nodes = dec.last_round_nodes()
            lg = dec.debug_logits()
            assert sorted(nd["heap"] for nd in nodes) == sorted(rounds[r])
            for i, nd in enumerate(nodes):
                o = rounds[r][nd["heap"]]
                worst = max(worst, float(np.max(np.abs(lg[i] - o.logits))))
                if o.margin > 0.1:
                    assert nd["token"] == o.token, (r, nd, o.token)
                    checked += 1
        assert worst < 5e-2 and checked > 0
    finally:
        dec.close()


def test_batch_invariance():
    dexlib = require_gpu()
    shape, X, T = SMALL, [1, 2, 3, 4], 10
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompts = di.gen_prompts(shape, 3, 50).tolist()
    outs = {}
    for batch in (1, 3):
        dec = dexlib.Decoder(shape, w, X, batch=batch, max_ctx=160, max_new=T)
        try:
            for b in range(batch):
                dec.prefill(b, prompts[b] if batch == 3 else prompts[1])
            outs[batch] = dec.generate()
        finally:
            dec.close()
    assert outs[1][0] == outs[3][1]

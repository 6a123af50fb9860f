"""GPU checks of the two split-K summations of the layer GEMMs and of the prefill passes.

* Exact fixed-point tile sums at L2 (decoders whose lattice gives a sequence at most 16
  nodes per round) and fp32 partial tiles in segment order (``DEX_SUM_FP32=1``): each is
  lossless (DEX tokens and final-depth logits equal the library's AR stream bit for bit)
  and within 5e-2 of the fp64 oracle; the two agree with each other to fp32 rounding.
* Prefill passes of other sizes and node groups (``DEX_PREFILL_ROWS``,
  ``DEX_PREFILL_GROUP_ROWS``): several passes and groups with a ragged tail decode to the
  oracle's stream.
* A partial outside the fixed-point range (weights scaled by 2^32) is reported as
  DEX_ERANGE by the round, again by the next round, and a fresh decoder is unaffected.
"""
import os

import numpy as np
import pytest

import dex_inputs as di
from gpu_util import check_logits_and_tokens, oracle_model, require_gpu
from oracle import dex as odex

pytestmark = pytest.mark.gpu

SMALL = di.ModelShape(n_layers=4, d_model=1024, n_heads=8, n_kv_heads=8, head_dim=128, d_ff=2816,
                      vocab=8192, tied_head=False)
TINY_UNTIED = di.ModelShape(**{**di.TINY.__dict__, "tied_head": False})


class _env:
    """Set environment variables for the decoders created inside the block (read at init)."""

    def __init__(self, **kv):
        self.kv = kv

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.kv}
        os.environ.update({k: str(v) for k, v in self.kv.items()})

    def __exit__(self, *exc):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _dex_and_ar(dexlib, shape, w, X, prompt, T, max_ctx=256):
    """DEX then AR from the same prompt: committed tokens and final-depth logits of each."""
    dec = dexlib.Decoder(shape, w, X, batch=1, max_ctx=max_ctx, max_new=T, debug_logits=True)
    out = {}
    try:
        for mode in ("dex", "ar"):
            dec.prefill(0, prompt)
            ys, zs = [], []
            while len(ys) < T:
                tok, nc = dec.step(ar=(mode == "ar"))
                if nc[0]:
                    nodes = dec.last_round_nodes()
                    want = len(X) - 1 if mode == "dex" else 0
                    k = [i for i, nd in enumerate(nodes) if nd["stage"] == want]
                    assert len(k) == 1
                    ys.append(tok[0])
                    zs.append(dec.debug_logits()[k[0]].copy())
            out[mode] = (ys, zs)
    finally:
        dec.close()
    (y_dex, z_dex), (y_ar, z_ar) = out["dex"], out["ar"]
    assert y_dex == y_ar
    for t in range(T):
        assert np.array_equal(z_dex[t].view(np.uint32), z_ar[t].view(np.uint32)), f"token {t}: logits differ"
    return y_ar, z_ar


def test_both_split_k_summations_are_lossless_and_match_the_oracle():
    dexlib = require_gpu()
    shape, X, T = SMALL, [1, 2, 3, 4], 12
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 40)[0].tolist()
    runs = {}
    for mode, env in (("fixed", {"DEX_SUM_FP32": "0"}), ("fp32", {"DEX_SUM_FP32": "1"})):
        with _env(**env):
            runs[mode] = _dex_and_ar(dexlib, shape, w, X, prompt, T)
    m = oracle_model(shape, w)
    for mode, (y, z) in runs.items():
        ref = odex.ar_generate(m, prompt, T, force=y)
        check_logits_and_tokens(z, y, ref)
    # the same model through either summation: logits agree to fp32 rounding up to the first
    # token where the two streams part (a near-tie may flip; after it the contexts differ)
    (ya, za), (yb, zb) = runs["fixed"], runs["fp32"]
    n = next((t for t in range(T) if ya[t] != yb[t]), T)
    d = max(float(np.max(np.abs(za[t] - zb[t]))) for t in range(max(1, n)))
    assert d < 1e-3, d


@pytest.mark.parametrize("rows,group", [(48, 16), (64, 64), (256, 128)])
def test_prefill_passes_and_groups(rows, group):
    dexlib = require_gpu()
    shape, X, T = TINY_UNTIED, [2, 4, 6, 8], 8
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 131)[0].tolist()   # 130 prefilled positions: passes + a ragged tail
    with _env(DEX_PREFILL_ROWS=rows, DEX_PREFILL_GROUP_ROWS=group):
        y, z = _dex_and_ar(dexlib, shape, w, X, prompt, T)
    ref = odex.ar_generate(oracle_model(shape, w), prompt, T, force=y)
    check_logits_and_tokens(z, y, ref)


def test_prefill_pass_settings_are_checked():
    dexlib = require_gpu()
    w = di.gen_weights(TINY_UNTIED, 0.3, seed=0, device="cuda")
    for env in ({"DEX_PREFILL_ROWS": 40}, {"DEX_PREFILL_GROUP_ROWS": 8}, {"DEX_PREFILL_ROWS": 256,
                                                                          "DEX_PREFILL_GROUP_ROWS": 16}):
        with _env(**env), pytest.raises(dexlib.DexError) as e:
            dexlib.Decoder(TINY_UNTIED, w, [2, 4, 6, 8], batch=1, max_ctx=64, max_new=4)
        assert e.value.code == dexlib.DEX_EINVAL


def test_out_of_range_partial_reports_erange():
    dexlib = require_gpu()
    shape, X = TINY_UNTIED, [2, 4, 6, 8]
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 20)[0].tolist()
    dec = dexlib.Decoder(shape, w, X, batch=1, max_ctx=64, max_new=6)
    try:
        dec.prefill(0, prompt)
        want = dec.generate()[0]
    finally:
        dec.close()
    big = dict(w)
    big["l0.wq"] = (w["l0.wq"].float() * 2.0 ** 32).to(w["l0.wq"].dtype)
    dec = dexlib.Decoder(shape, big, X, batch=1, max_ctx=64, max_new=6)
    try:
        for _ in range(2):   # reported by the round, and again (the state was reset, not stuck)
            dec.prefill(0, prompt)
            with pytest.raises(dexlib.DexError) as e:
                dec.generate()
            assert e.value.code == dexlib.DEX_ERANGE
    finally:
        dec.close()
    dec = dexlib.Decoder(shape, w, X, batch=1, max_ctx=64, max_new=6)
    try:
        dec.prefill(0, prompt)
        assert dec.generate()[0] == want
    finally:
        dec.close()


def test_prefill_fallback_for_three_query_heads_per_kv_head():
    """Twelve query heads on four KV heads: 128 is not a multiple of 3, so prefill passes
    take the lattice attention kernel (items of five rows, fifteen queries per pass); the
    decode is lossless and matches the oracle."""
    dexlib = require_gpu()
    shape = di.ModelShape(n_layers=4, d_model=768, n_heads=12, n_kv_heads=4, head_dim=64, d_ff=2048,
                          vocab=4096, tied_head=False)
    X, T = [1, 2, 3, 4], 10
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 150)[0].tolist()
    y, z = _dex_and_ar(dexlib, shape, w, X, prompt, T)
    ref = odex.ar_generate(oracle_model(shape, w), prompt, T, force=y)
    check_logits_and_tokens(z, y, ref)

"""GPU edge cases of the DEX path: degenerate exploration sets and models, empty and
ragged prompts, the largest supported context, and host-side argument errors.

Each decode case checks the lossless invariant (DEX tokens and final-depth logits equal
the library's AR stream bit for bit); the oracle comparisons use the fp64 oracle.
"""
import numpy as np
import pytest

import dex_inputs as di
from gpu_util import check_logits_and_tokens, oracle_model, require_gpu
from oracle import dex as odex

pytestmark = pytest.mark.gpu

SMALL = di.ModelShape(n_layers=4, d_model=1024, n_heads=8, n_kv_heads=8, head_dim=128, d_ff=2816,
                      vocab=8192, tied_head=False)
TINY_UNTIED = di.ModelShape(**{**di.TINY.__dict__, "tied_head": False})


def _run(dexlib, shape, w, X, prompts, T, max_ctx, sample=False, debug_logits=True):
    """DEX then AR on the same prompts; per sequence tokens and final-depth logits."""
    B, N = len(prompts), len(X)
    dec = dexlib.Decoder(shape, w, X, batch=B, max_ctx=max_ctx, max_new=T, sample=sample, tau=0.7, seed=5,
                         debug_logits=debug_logits)
    out = {}
    try:
        for mode in ("dex", "ar"):
            for b, p in enumerate(prompts):
                dec.prefill(b, p)
            dec.reset_stats()
            ys, zs = [[] for _ in range(B)], [[] for _ in range(B)]
            while min(len(y) for y in ys) < T:
                tok, nc = dec.step(ar=(mode == "ar"))
                nodes = dec.last_round_nodes()
                lg = dec.debug_logits() if debug_logits else None
                for b in range(B):
                    if nc[b]:
                        want = N - 1 if mode == "dex" else 0
                        k = [i for i, nd in enumerate(nodes) if nd["seq"] == b and nd["stage"] == want]
                        assert len(k) == 1
                        ys[b].append(tok[b])
                        if debug_logits:
                            zs[b].append(lg[k[0]].copy())
            out[mode] = (ys, zs, dec.stats())
    finally:
        dec.close()
    for b in range(B):
        assert out["dex"][0][b] == out["ar"][0][b], f"sequence {b}: DEX tokens differ from AR"
        for t, (za, zb) in enumerate(zip(out["dex"][1][b], out["ar"][1][b])):
            assert np.array_equal(za.view(np.uint32), zb.view(np.uint32)), f"sequence {b} token {t}"
    return out


def test_single_exit_depth_is_plain_ar():
    """X = {L}: one stage, every round commits its only node (k* = 0), no branch KV."""
    dexlib = require_gpu()
    w = di.gen_weights(TINY_UNTIED, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(TINY_UNTIED, 1, 20)[0].tolist()
    out = _run(dexlib, TINY_UNTIED, w, [8], [prompt], 12, 64)
    st = out["dex"][2]
    assert st["rounds"] == 12 and st["commits"] == 12 and st["kstar_hist"][0] == 12


def test_all_depths_agree_collapses_to_shallowest():
    """alpha = 0: every residual branch is zero, the hidden state stays the embedding and
    every depth predicts the same token, so each commit keeps the shallowest anchor (k* = 0);
    tokens and round count equal the oracle's Algorithm 1."""
    dexlib = require_gpu()
    shape, X, T = TINY_UNTIED, [2, 4, 6, 8], 10
    w = di.gen_weights(shape, 0.0, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 16)[0].tolist()
    out = _run(dexlib, shape, w, X, [prompt], T, 64)
    st = out["dex"][2]
    assert st["kstar_hist"][0] == T
    m = oracle_model(shape, w)
    ref = odex.dex_generate(m, prompt, X, T)
    assert out["dex"][0][0] == ref.tokens
    assert st["rounds"] == ref.rounds


def test_prompt_of_one_token():
    """Nothing to prefill: the first round's stage-0 node is at position 0."""
    dexlib = require_gpu()
    shape, X, T = TINY_UNTIED, [2, 4, 6, 8], 10
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = [int(di.gen_prompts(shape, 1, 1)[0, 0])]
    out = _run(dexlib, shape, w, X, [prompt], T, 64)
    m = oracle_model(shape, w)
    y, z = out["ar"][0][0], out["ar"][1][0]
    ref = odex.ar_generate(m, prompt, T, force=y)
    check_logits_and_tokens(z, y, ref)


def test_ragged_batch_matches_single_sequences():
    """Prompts of 1, 130 and 257 tokens (ragged 128-key groups and prefill chunks) in one
    batch decode exactly as each does alone (greedy: Gumbel rows are keyed by the
    sequence index, so sampled streams legitimately differ between batch slots)."""
    dexlib = require_gpu()
    shape, X, T = SMALL, [1, 2, 3, 4], 8
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompts = [di.gen_prompts(shape, 1, n, seed=40 + n)[0].tolist() for n in (1, 130, 257)]
    batch = _run(dexlib, shape, w, X, prompts, T, 300)
    for b, p in enumerate(prompts):
        alone = _run(dexlib, shape, w, X, [p], T, 300)
        assert alone["dex"][0][0] == batch["dex"][0][b]
        for za, zb in zip(alone["dex"][1][0], batch["dex"][1][b]):
            assert np.array_equal(za.view(np.uint32), zb.view(np.uint32))


def test_largest_context():
    """max_ctx = 4096 (32 key groups, the attention kernel's limit), filled to the last
    position: prompt + new tokens + N = max_ctx.  Oracle parity on the last tokens."""
    dexlib = require_gpu()
    shape, X, T = SMALL, [1, 2, 3, 4], 6
    max_ctx = 4096
    P = max_ctx - T - len(X)
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, P, seed=9)[0].tolist()
    out = _run(dexlib, shape, w, X, [prompt], T, max_ctx)
    m = oracle_model(shape, w)
    y, z = out["ar"][0][0], out["ar"][1][0]
    ref = odex.ar_generate(m, prompt, T, force=y)
    err, checked = check_logits_and_tokens(z, y, ref)
    assert checked >= 1


def test_argument_and_state_errors():
    """Host-side checks return status codes before any launch; the handle stays usable."""
    dexlib = require_gpu()
    shape, X = TINY_UNTIED, [2, 4, 6, 8]
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    dec = dexlib.Decoder(shape, w, X, batch=2, max_ctx=64, max_new=8)
    try:
        with pytest.raises(dexlib.DexError) as e:
            dec.step()                                  # nothing prefilled
        assert e.value.code == dexlib.DEX_ESTATE
        with pytest.raises(dexlib.DexError) as e:
            dec.prefill(0, [1] * 60)                    # 60 + 8 + 4 > 64
        assert e.value.code == dexlib.DEX_ECAPACITY
        with pytest.raises(dexlib.DexError) as e:
            dec.prefill(2, [1, 2])                      # no such sequence
        assert e.value.code == dexlib.DEX_EINVAL
        with pytest.raises(dexlib.DexError) as e:
            dec.prefill(0, [shape.vocab])               # token out of range
        assert e.value.code == dexlib.DEX_EINVAL
        dec.prefill(0, [1, 2, 3])
        tok, nc = dec.step()
        assert nc[1] == 0
        with pytest.raises(dexlib.DexError) as e:
            dec.step(ar=True)                           # sequence 0 is mid-way through DEX
        assert e.value.code == dexlib.DEX_ESTATE
        out = dec.generate()
        assert len(out[0]) == 8 and all(0 <= t < shape.vocab for t in out[0])
    finally:
        dec.close()
    with pytest.raises(dexlib.DexError):
        dexlib.Decoder(shape, w, [2, 4, 6], batch=1, max_ctx=64, max_new=8)   # X must end at L
    with pytest.raises(dexlib.DexError):
        dexlib.Decoder(shape, w, X, batch=1, max_ctx=4097, max_new=8)          # above the context cap


@pytest.mark.parametrize("sample", [False, True])
def test_vanilla_lattice_without_decs_matches_oracle(sample):
    """decs = 0 (every node decoded on its own, section 4's vanilla ablation): still lossless,
    and every round's nodes, tokens and the round count equal the oracle's Algorithm 1
    run without DECS."""
    dexlib = require_gpu()
    shape, X, T = TINY_UNTIED, [2, 4, 6, 8], 12
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 24)[0].tolist()
    dec = dexlib.Decoder(shape, w, X, batch=1, max_ctx=64, max_new=T, sample=sample, tau=0.7, seed=5, decs=False,
                         debug_logits=True)
    m = oracle_model(shape, w)
    rule = odex.Rule(sample=sample, tau=0.7, seed=5)
    ref = odex.dex_generate(m, prompt, X, T, rule=rule, use_decs=False, keep_logits=True)
    rounds = {}
    for nd in ref.nodes:
        rounds.setdefault(nd.round, {})[nd.node] = nd
    try:
        dec.prefill(0, prompt)
        toks, checked = [], 0
        for r in range(ref.rounds):
            tok, nc = dec.step()
            if nc[0]:
                toks.append(tok[0])
            nodes = dec.last_round_nodes()
            assert sorted(nd["heap"] for nd in nodes) == sorted(rounds[r])
            for nd in nodes:
                o = rounds[r][nd["heap"]]
                if o.margin > 0.1:
                    assert nd["token"] == o.token
                    checked += 1
        assert toks == ref.tokens and checked > 0
        assert dec.stats()["rounds"] == ref.rounds
    finally:
        dec.close()


def test_single_exit_variant_and_ten_stages():
    """X = {d_0, L} (one intermediate exit: the single-exit variant) and |X| = 10 (the
    largest exploration set) on a 10-layer model: lossless against the library's AR path
    and the oracle's Algorithm 1 token stream."""
    dexlib = require_gpu()
    shape = di.ModelShape(**{**TINY_UNTIED.__dict__, "n_layers": 10})
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 20)[0].tolist()
    m = oracle_model(shape, w)
    for X in ([3, 10], list(range(1, 11))):
        T = 8
        out = _run(dexlib, shape, w, X, [prompt], T, 64)
        ref = odex.dex_generate(m, prompt, X, T)
        assert out["dex"][0][0] == ref.tokens
        assert out["dex"][2]["rounds"] == ref.rounds


def test_batch_of_sixteen_sequences():
    """16 independent sequences with different prompt lengths in one handle: each equals
    its own AR stream bit for bit (greedy)."""
    dexlib = require_gpu()
    shape, X, T = TINY_UNTIED, [2, 4, 6, 8], 6
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompts = [di.gen_prompts(shape, 1, 5 + 3 * b, seed=100 + b)[0].tolist() for b in range(16)]
    _run(dexlib, shape, w, X, prompts, T, 64)


@pytest.mark.parametrize("cap", [1, 2])
def test_sparse_lattice_on_gpu(cap):
    """max_branch caps the speculation depth: DEX is still bit-identical to AR, and every
    round's nodes and tokens equal the oracle's capped Algorithm 1."""
    dexlib = require_gpu()
    shape, X, T = TINY_UNTIED, [1, 2, 3, 4, 5, 6, 7, 8], 10
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 24)[0].tolist()
    dec = dexlib.Decoder(shape, w, X, batch=1, max_ctx=64, max_new=T, debug_logits=True, max_branch=cap)
    m = oracle_model(shape, w)
    ref = odex.dex_generate(m, prompt, X, T, max_branch=cap)
    rounds = {}
    for nd in ref.nodes:
        rounds.setdefault(nd.round, {})[nd.node] = nd
    try:
        dec.prefill(0, prompt)
        toks, checked = [], 0
        for r in range(ref.rounds):
            tok, nc = dec.step()
            if nc[0]:
                toks.append(tok[0])
            nodes = dec.last_round_nodes()
            assert sorted(nd["heap"] for nd in nodes) == sorted(rounds[r])
            for nd in nodes:
                o = rounds[r][nd["heap"]]
                if o.margin > 0.1:
                    assert nd["token"] == o.token
                    checked += 1
        assert toks == ref.tokens and checked > 0
        dec.prefill(0, prompt)
        y_ar = dec.generate(ar=True)[0]
        assert y_ar == toks
    finally:
        dec.close()


@pytest.mark.parametrize("which,sample", [("tiny", False), ("tiny", True), ("small", False)])
def test_inducing_adapters_on_gpu(which, sample):
    """Inducing adapters at the non-final exits (Appendix C.2, gate 2.0): every round's nodes
    and exit logits equal the oracle's adapted Algorithm 1, the committed stream is still
    bit-identical to AR, and the adapters move the intermediate logits by far more than the
    tolerance (so the comparison could tell adapted from plain exits apart)."""
    from oracle.model import widen_bf16
    dexlib = require_gpu()
    shape, X, T = (TINY_UNTIED, [2, 4, 6, 8], 10) if which == "tiny" else (SMALL, [1, 2, 3, 4], 8)
    w = di.gen_weights(shape, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(shape, 1, 24)[0].tolist()
    ads = di.gen_adapters(shape, X, gate=2.0, device="cuda")
    wide = [{k: (v if k == "alpha" else widen_bf16(di.bf16_bits(v))) for k, v in a.items()} for a in ads]
    m = oracle_model(shape, w)
    rule = odex.Rule(sample=sample, tau=0.7, seed=5)
    ref = odex.dex_generate(m, prompt, X, T, rule=rule, adapters=wide, keep_logits=True)
    plain = odex.dex_generate(m, prompt, X, T, rule=rule, keep_logits=True)
    first_plain = {(nd.round, nd.node): nd for nd in plain.nodes if nd.round < len(X)}
    moved = max(float(np.max(np.abs(nd.logits - first_plain[(nd.round, nd.node)].logits)))
                for nd in ref.nodes if nd.round < len(X) and nd.stage < len(X) - 1)
    assert moved > 0.25
    rounds = {}
    for nd in ref.nodes:
        rounds.setdefault(nd.round, {})[nd.node] = nd
    dec = dexlib.Decoder(shape, w, X, batch=1, max_ctx=64, max_new=T, sample=sample, tau=0.7, seed=5,
                         debug_logits=True, adapters=ads)
    try:
        dec.prefill(0, prompt)
        toks, checked, worst = [], 0, 0.0
        for r in range(ref.rounds):
            tok, nc = dec.step()
            if nc[0]:
                toks.append(tok[0])
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
        assert toks == ref.tokens
        dec.prefill(0, prompt)
        assert dec.generate(ar=True)[0] == toks
    finally:
        dec.close()

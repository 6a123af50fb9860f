"""Pins for oracle/model.py against torch library routines and closed forms (fp64, CPU)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from conftest import tiny_model
from oracle import model as M

rng = np.random.default_rng(0)


def test_widen_bf16_exact():
    x = torch.randn(1000, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(M.widen_bf16(bits), x.double().numpy())


def test_rmsnorm_matches_torch():
    x = rng.standard_normal((5, 64))
    g = rng.standard_normal(64)
    ref = F.rms_norm(torch.tensor(x), (64,), weight=torch.tensor(g), eps=1e-5).numpy()
    assert np.allclose(M.rmsnorm(x, g, 1e-5), ref, rtol=1e-12, atol=1e-12)


def test_silu_matches_torch():
    x = rng.standard_normal(1000) * 5
    assert np.allclose(M.silu(x), F.silu(torch.tensor(x)).numpy(), rtol=1e-12, atol=1e-14)


def test_rope_closed_form_two_dims():
    # head_dim 2: the pair (x0, x1) rotates by angle pos * theta^0 = pos radians
    x = np.array([[[1.0, 0.0]], [[0.0, 1.0]], [[3.0, 4.0]]])
    pos = np.array([0.7, 2.0, -1.3])
    out = M.rope(x, pos, 10000.0)
    for i in range(3):
        c, s = np.cos(pos[i]), np.sin(pos[i])
        want = np.array([c * x[i, 0, 0] - s * x[i, 0, 1], s * x[i, 0, 0] + c * x[i, 0, 1]])
        assert np.allclose(out[i, 0], want, atol=1e-15)


def test_rope_frequencies_and_pairs():
    # hd = 8: component j pairs with j + 4 and rotates at theta^(-2j/8)
    hd, theta = 8, 100.0
    for j in range(4):
        x = np.zeros((1, 1, hd))
        x[0, 0, j] = 1.0
        out = M.rope(x, np.array([3.0]), theta)[0, 0]
        ang = 3.0 * theta ** (-2.0 * j / hd)
        want = np.zeros(hd)
        want[j], want[j + 4] = np.cos(ang), np.sin(ang)
        assert np.allclose(out, want, atol=1e-15)


def test_rope_relative_position_and_norm():
    q = rng.standard_normal((1, 2, 16))
    k = rng.standard_normal((1, 2, 16))
    d1 = np.sum(M.rope(q, np.array([10]), 1e4) * M.rope(k, np.array([3]), 1e4))
    d2 = np.sum(M.rope(q, np.array([107]), 1e4) * M.rope(k, np.array([100]), 1e4))
    assert d1 == pytest.approx(d2, rel=1e-10)
    assert np.allclose(np.linalg.norm(M.rope(q, np.array([55]), 1e4), axis=-1), np.linalg.norm(q, axis=-1))


@pytest.mark.parametrize("H,KVH", [(4, 4), (8, 2)])
def test_causal_attention_matches_sdpa(H, KVH):
    n, ctx, hd = 5, 9, 16
    q = rng.standard_normal((n, H, hd))
    k = rng.standard_normal((ctx, KVH, hd))
    v = rng.standard_normal((ctx, KVH, hd))
    qpos = np.arange(ctx - n, ctx)
    out = M.causal_attention(q, k, v, qpos)
    tq = torch.tensor(q).permute(1, 0, 2)[None]                                 # [1,H,n,hd]
    tk = torch.tensor(k).permute(1, 0, 2).repeat_interleave(H // KVH, 0)[None]   # [1,H,ctx,hd]
    tv = torch.tensor(v).permute(1, 0, 2).repeat_interleave(H // KVH, 0)[None]
    mask = torch.tensor(np.arange(ctx)[None, :] <= qpos[:, None])
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)[0].permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


def _torch_reference_forward(shape, w, tokens, depth):
    """Independent full-sequence restatement with torch library routines (fp64)."""
    t = lambda k: w[k].double()
    h = t("embed")[torch.tensor(tokens, dtype=torch.long)]
    n = len(tokens)
    H, KVH, hd = shape.n_heads, shape.n_kv_heads, shape.head_dim
    half = hd // 2
    inv = shape.rope_theta ** (-(2.0 * torch.arange(half, dtype=torch.float64)) / hd)
    ang = torch.arange(n, dtype=torch.float64)[:, None] * inv[None]
    cos, sin = torch.cos(ang)[:, None], torch.sin(ang)[:, None]

    def rot(x):
        return torch.cat([x[..., :half] * cos - x[..., half:] * sin, x[..., half:] * cos + x[..., :half] * sin], -1)
    for l in range(depth):
        a = F.rms_norm(h, (shape.d_model,), weight=t(f"l{l}.attn_norm"), eps=shape.rms_eps)
        q = rot(F.linear(a, t(f"l{l}.wq")).view(n, H, hd)).transpose(0, 1)
        k = rot(F.linear(a, t(f"l{l}.wk")).view(n, KVH, hd)).transpose(0, 1)
        v = F.linear(a, t(f"l{l}.wv")).view(n, KVH, hd).transpose(0, 1)
        o = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True, enable_gqa=True)[0]
        h = h + F.linear(o.transpose(0, 1).reshape(n, H * hd), t(f"l{l}.wo"))
        b = F.rms_norm(h, (shape.d_model,), weight=t(f"l{l}.ffn_norm"), eps=shape.rms_eps)
        h = h + F.linear(F.silu(F.linear(b, t(f"l{l}.wg"))) * F.linear(b, t(f"l{l}.wu")), t(f"l{l}.wd"))
    head = t("embed") if shape.tied_head else t("lm_head")
    return F.linear(F.rms_norm(h, (shape.d_model,), weight=t("final_norm"), eps=shape.rms_eps), head).numpy()


@pytest.mark.parametrize("alpha,tied", [(0.1, True), (1.0, False)])
def test_decoder_matches_torch_restatement(alpha, tied):
    shape, w, m = tiny_model(alpha, tied)
    tokens = [5, 77, 4000, 12, 12, 901, 3]
    cache = m.new_cache(16)
    h = m.forward(tokens, 0, cache)
    ref = _torch_reference_forward(shape, w, tokens, shape.n_layers)
    assert np.allclose(m.exit_logits(h), ref, rtol=1e-9, atol=1e-9)


def test_incremental_decode_equals_full_sequence():
    shape, w, m = tiny_model(1.0, False)
    tokens = [9, 8, 7, 6, 5, 4, 3, 2]
    full = m.forward(tokens, 0, m.new_cache(16))
    cache = m.new_cache(16)
    rows = [m.forward(tokens[:3], 0, cache)]
    for p in range(3, len(tokens)):
        rows.append(m.forward([tokens[p]], p, cache))
    inc = np.concatenate(rows)
    assert np.allclose(inc, full, rtol=1e-11, atol=1e-12)


def test_gqa_decoder_matches_torch_restatement():
    import dex_inputs as di
    shape = di.ModelShape(n_layers=2, d_model=128, n_heads=8, n_kv_heads=2, head_dim=16, d_ff=96,
                          vocab=300, tied_head=False, rope_theta=1e6)
    w = di.gen_weights(shape, 0.5, seed=4)
    m = M.OracleModel(shape, {k: di.bf16_bits(v) for k, v in w.items()}, keep_widened=False)
    tokens = [1, 299, 17, 4, 4]
    h = m.forward(tokens, 0, m.new_cache(8))
    ref = _torch_reference_forward(shape, w, tokens, shape.n_layers)
    assert np.allclose(m.exit_logits(h), ref, rtol=1e-9, atol=1e-9)


def test_intermediate_depth_exit_uses_shared_head():
    shape, w, m = tiny_model(1.0, False)
    tokens = [3, 1, 4, 1, 5]
    hist = m.forward(tokens, 0, m.new_cache(8), keep_depths=True)
    for depth in (2, 5, 8):
        ref = _torch_reference_forward(shape, w, tokens, depth)
        assert np.allclose(m.exit_logits(hist[depth - 1]), ref, rtol=1e-9, atol=1e-9)

"""Plain fp64 Llama-style decoder and shared exit head -- oracle side.

The model "Depth Exploration for LLM Decoding" runs DEX on (section 4: Llama-2,
CodeLlama, Qwen3 decoders; Appendix C.2: intermediate depths are decoded "by the
same final normalization and LM head as the backbone").  The pages do not print
the block, so the plain Llama reading is taken:

    x_0 = E[token]
    per layer:  a = RMSNorm(h; g_attn)
                q, k, v = a W_q^T, a W_k^T, a W_v^T          (rows [out][in])
                q, k = RoPE(q, pos), RoPE(k, pos)               (rotate-half pairs j, j+hd/2)
                o = softmax(q k^T / sqrt(hd)) v  over keys at positions 0..pos
                    (query head h reads key/value head h // (n_heads / n_kv_heads))
                h = h + o W_o'^T                                (W_o' = alpha W_o, pre-folded)
                b = RMSNorm(h; g_ffn)
                h = h + (SiLU(b W_g^T) * (b W_u^T)) W_d'^T     (W_d' = alpha W_d, pre-folded)
    exit at depth l:  z_l = RMSNorm(h_l; g_final) W_lm^T

RMSNorm(x; g) = x / sqrt(mean(x^2) + eps) * g.  RoPE frequencies theta^(-2j/hd).
Weights arrive as bf16 bit patterns and are widened exactly to fp64; all arithmetic
is fp64.  TEST INFRASTRUCTURE ONLY.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> fp64: a bf16 pattern is the top half of an fp32 pattern."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE.  x: [n, heads, hd]; pos: [n] absolute positions."""
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]   # [n, half]
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, qpos: np.ndarray) -> np.ndarray:
    """softmax(q k^T / sqrt(hd)) v with keys at positions 0..ctx-1 and a causal mask.

    q: [n, H, hd] queries at absolute positions qpos [n]; k, v: [ctx, KVH, hd] keys and
    values at positions 0..ctx-1.  Query head h reads key/value head h // (H / KVH).
    Key c is visible to the query at position p iff c <= p.
    """
    n, H, hd = q.shape
    ctx, KVH, _ = k.shape
    group = H // KVH
    kk = np.repeat(k, group, axis=1)                        # [ctx, H, hd]
    vv = np.repeat(v, group, axis=1)
    s = np.einsum("nhd,chd->hnc", q, kk) / np.sqrt(hd)       # [H, n, ctx]
    visible = np.arange(ctx)[None, :] <= np.asarray(qpos)[:, None]   # [n, ctx]
    s = np.where(visible[None], s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return np.einsum("hnc,chd->nhd", p, vv)


class KVCache:
    """Per-layer key/value rows indexed by absolute position (fp64)."""

    def __init__(self, n_layers: int, max_ctx: int, n_kv_heads: int, head_dim: int):
        self.k = np.zeros((n_layers, max_ctx, n_kv_heads, head_dim))
        self.v = np.zeros((n_layers, max_ctx, n_kv_heads, head_dim))


class OracleModel:
    """fp64 decoder over widened bf16 weights.  ``weights``: name -> uint16 bit array.

    With ``keep_widened=False`` each layer's weights are widened on every use instead
    of being held as fp64 (8 bytes per parameter), for models too large for host RAM.
    """

    def __init__(self, shape, weights: Dict[str, np.ndarray], keep_widened: bool = True):
        self.shape = shape
        self.L = shape.n_layers
        self.eps = shape.rms_eps
        self.theta = shape.rope_theta
        self.keep_widened = keep_widened
        self.embed_bits = weights["embed"]
        self.final_norm = widen_bf16(weights["final_norm"])
        self.lm_head = None
        if keep_widened:
            self.lm_head = widen_bf16(weights["embed" if shape.tied_head else "lm_head"])
        self.lm_head_bits = weights["embed" if shape.tied_head else "lm_head"]
        self.layer_bits = [{n: weights[f"l{l}.{n}"] for n in LAYER_TENSORS} for l in range(self.L)]
        self.layers: List[Optional[Dict[str, np.ndarray]]] = [None] * self.L
        if keep_widened:
            for l in range(self.L):
                self.layers[l] = {n: widen_bf16(b) for n, b in self.layer_bits[l].items()}

    def _weights(self, l: int) -> Dict[str, np.ndarray]:
        if self.layers[l] is not None:
            return self.layers[l]
        return {n: widen_bf16(b) for n, b in self.layer_bits[l].items()}

    def _lm_head(self) -> np.ndarray:
        return self.lm_head if self.lm_head is not None else widen_bf16(self.lm_head_bits)

    def new_cache(self, max_ctx: int) -> KVCache:
        s = self.shape
        return KVCache(self.L, max_ctx, s.n_kv_heads, s.head_dim)

    # -- one decoder layer over a run of consecutive positions -----------------------
    def layer(self, l: int, h: np.ndarray, pos0: int, cache: KVCache) -> np.ndarray:
        """Apply layer l (0-based) to rows h [n, d] at positions pos0 .. pos0+n-1.

        Writes the rows' keys/values into ``cache`` first; query at position p then
        attends every cached key at positions 0..p (causal).
        """
        s, W = self.shape, self._weights(l)
        n = h.shape[0]
        hd, H, KVH = s.head_dim, s.n_heads, s.n_kv_heads
        pos = np.arange(pos0, pos0 + n)
        a = rmsnorm(h, W["attn_norm"], self.eps)
        q = (a @ W["wq"].T).reshape(n, H, hd)
        k = (a @ W["wk"].T).reshape(n, KVH, hd)
        v = (a @ W["wv"].T).reshape(n, KVH, hd)
        q, k = rope(q, pos, self.theta), rope(k, pos, self.theta)
        cache.k[l, pos0:pos0 + n] = k
        cache.v[l, pos0:pos0 + n] = v
        o = np.empty((n, H, hd))
        for c0 in range(0, n, 128):      # query blocks bound the [H, n, ctx] score array
            c1 = min(n, c0 + 128)
            ctx = pos0 + c1
            o[c0:c1] = causal_attention(q[c0:c1], cache.k[l, :ctx], cache.v[l, :ctx], pos[c0:c1])
        h = h + o.reshape(n, H * hd) @ W["wo"].T
        b = rmsnorm(h, W["ffn_norm"], self.eps)
        h = h + (silu(b @ W["wg"].T) * (b @ W["wu"].T)) @ W["wd"].T
        return h

    def forward(self, tokens: Sequence[int], pos0: int, cache: KVCache, depth: Optional[int] = None,
                keep_depths: bool = False):
        """Run tokens at positions pos0.. through layers 1..depth (default L).

        Returns the hidden rows after layer ``depth``, or, with keep_depths, the list
        [h after layer 1, ..., h after layer depth].
        """
        depth = self.L if depth is None else depth
        h = widen_bf16(self.embed_bits[np.asarray(tokens, dtype=np.int64)])
        hist = []
        for l in range(depth):
            h = self.layer(l, h, pos0, cache)
            if keep_depths:
                hist.append(h)
        return hist if keep_depths else h

    def exit_logits(self, h: np.ndarray, adapter: Optional[Dict] = None) -> np.ndarray:
        """Shared exit head: RMSNorm(h; g_final) W_lm^T (Appendix C.2), after the inducing
        adapter of the depth when one is given."""
        if adapter is not None:
            h = apply_adapter(h, adapter, self.eps)
        return rmsnorm(h, self.final_norm, self.eps) @ self._lm_head().T


def silu_act(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def apply_adapter(h: np.ndarray, ad: Dict, eps: float) -> np.ndarray:
    """Inducing adapter of Appendix C.2 at a non-final depth:

        delta = alpha (W2 sigma(W1 RMSNorm(h; g) + b1) + b2),   h~ = h + delta,

    two linear layers with biases (hidden width m = 2h), the backbone activation sigma
    (SiLU for these SwiGLU decoders) and the scalar gate alpha.  ``ad`` holds widened fp64
    arrays g, w1 [m][h], b1 [m], w2 [h][m], b2 [h] and the float alpha."""
    n = rmsnorm(h, ad["g"], eps)
    u = n @ ad["w1"].T + ad["b1"]
    return h + ad["alpha"] * (silu_act(u) @ ad["w2"].T + ad["b2"])

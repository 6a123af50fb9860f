"""Seeded synthetic inputs for Depth Exploration Decoding (DEX) workloads.

This module is the ONLY code shared by the CPU oracle (``oracle/``) and the
CUDA library (``lossless_depth_adaptive_gb300``): it produces model weights,
prompts and micro-benchmark inputs from seeds, and holds none of the method's
arithmetic (no normalisation, attention, exit head, sampling or lattice logic).

Workload shapes follow "Depth Exploration for LLM Decoding" (arXiv 2606.29223),
section 4 (decoder-only LLMs, batch 1, greedy or temperature sampling) with the
model sizes replaced by seeded synthetic stand-ins, because no trained weights
or datasets are available: prompts are uniform random token ids, weights are
approximately N(0, std) with the residual-branch outputs scaled by ``alpha``.

Determinism across devices
--------------------------
Every value is a pure function of (seed, tensor id, element index), computed
with 64-bit integer arithmetic that never overflows (a 32-bit value times a
multiplier below 2**31), followed by one exact int->float conversion and
correctly rounded float32 multiplies, then round-to-nearest-even to bfloat16.
The same call therefore yields bit-identical tensors on the CPU and on a GPU,
so the oracle can be fed the exact weights the library runs on.

The normal approximation is the Irwin-Hall sum of four independent 16-bit
uniforms (bounded to about +-3.46 sigma, excess kurtosis -0.3), which is
adequate for synthetic weights.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional

import torch

MASK32 = 0xFFFFFFFF
# Irwin-Hall(4) of 16-bit uniforms: mean 4*(65535/2), std 65536/sqrt(3) (to float precision).
_IH_MEAN = 131070
_IH_STD = math.sqrt((65536.0 * 65536.0 - 1.0) / 3.0)


@dataclass(frozen=True)
class ModelShape:
    """Shape of a Llama-style decoder (pre-norm, RMSNorm, RoPE, SwiGLU, no biases)."""
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    tied_head: bool
    rope_theta: float = 10000.0
    rms_eps: float = 1e-5


@dataclass(frozen=True)
class Workload:
    """One decoding workload: a model shape, its synthetic weights and a decode setup."""
    name: str
    shape: ModelShape
    alpha: float                 # residual-branch scale, folded into W_o and W_down
    X: List[int]                 # exploration set {d_0 < ... < d_{N-1} = L}
    batch: int
    prompt_len: int
    max_new: int
    sample: bool = False
    tau: float = 1.0
    decs: bool = True
    weight_seed: int = 0
    prompt_seed: int = 1
    gumbel_seed: int = 2
    weight_std: float = 0.02


TINY = ModelShape(n_layers=8, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64,
                  d_ff=688, vocab=4096, tied_head=True)
LLAMA7B = ModelShape(n_layers=32, d_model=4096, n_heads=32, n_kv_heads=32, head_dim=128,
                     d_ff=11008, vocab=32000, tied_head=False)
QWEN8B = ModelShape(n_layers=36, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128,
                    d_ff=12288, vocab=151936, tied_head=False, rope_theta=1e6)

WORKLOADS: Dict[str, Workload] = {
    # 8-layer tiny model: correctness reference.
    "tiny": Workload("tiny", TINY, alpha=0.1, X=[2, 4, 6, 8], batch=1,
                     prompt_len=32, max_new=64),
    # Llama-2-7B-shaped model, four explored depths, greedy.
    "llama7b_x4": Workload("llama7b_x4", LLAMA7B, alpha=0.05, X=[8, 16, 24, 32], batch=1,
                           prompt_len=512, max_new=256),
    # Same shape, eight explored depths, temperature-0.7 sampling with DECS.
    "llama7b_x8_sample": Workload("llama7b_x8_sample", LLAMA7B, alpha=0.05,
                                  X=list(range(4, 33, 4)), batch=1, prompt_len=1024,
                                  max_new=256, sample=True, tau=0.7),
    # Qwen3-8B-shaped GQA model, batch of 8 independent sequences.
    "qwen8b_x4_b8": Workload("qwen8b_x4_b8", QWEN8B, alpha=0.05, X=[9, 18, 27, 36], batch=8,
                             prompt_len=2048, max_new=128),
}


def workload(name: str, **overrides) -> Workload:
    """Return a named workload, optionally with fields replaced (e.g. alpha, X, max_new)."""
    w = WORKLOADS[name]
    if "shape" in overrides and isinstance(overrides["shape"], dict):
        overrides["shape"] = replace(w.shape, **overrides["shape"])
    return replace(w, **overrides)


# ----------------------------------------------------------------------------------------
# counter-based hash (own design: xor-shift / odd-multiply finaliser on 32-bit lanes)
# ----------------------------------------------------------------------------------------

def _mix32_int(x: int) -> int:
    x &= MASK32
    x = ((x ^ (x >> 16)) * 0x7FEB352D) & MASK32
    x = ((x ^ (x >> 15)) * 0x68E31DA5) & MASK32
    return x ^ (x >> 16)


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = x & MASK32
    x = ((x ^ (x >> 16)) * 0x7FEB352D) & MASK32
    x = ((x ^ (x >> 15)) * 0x68E31DA5) & MASK32
    return x ^ (x >> 16)


def _keys(seed: int, tensor_id: int):
    k1 = _mix32_int((seed * 0x9E3779B1) ^ _mix32_int(tensor_id + 0x632BE5AB))
    k2 = _mix32_int(k1 ^ 0x85EBCA6B ^ (seed >> 32))
    return k1, k2


def _hash_pair(idx: torch.Tensor, k1: int, k2: int):
    a = _mix32(_mix32(idx ^ k1) ^ k2)
    b = _mix32(a ^ k1 ^ 0x5BD1E995)
    return a, b


_CHUNK = 1 << 24


def _normal_fp32(numel: int, seed: int, tensor_id: int, std: float, scale: float,
                 device) -> torch.Tensor:
    """fp32 values ~ N(0, std) * scale, exactly reproducible on any device."""
    assert numel < (1 << 32)
    k1, k2 = _keys(seed, tensor_id)
    c = torch.tensor(std / _IH_STD, dtype=torch.float32, device=device)
    s = torch.tensor(scale, dtype=torch.float32, device=device)
    out = torch.empty(numel, dtype=torch.float32, device=device)
    for lo in range(0, numel, _CHUNK):
        hi = min(numel, lo + _CHUNK)
        idx = torch.arange(lo, hi, dtype=torch.int64, device=device)
        a, b = _hash_pair(idx, k1, k2)
        ih = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16) - _IH_MEAN
        v = ih.to(torch.float32) * c
        if scale != 1.0:
            v = v * s
        out[lo:hi] = v
    return out


def normal_bf16(shape, seed: int, tensor_id: int, std: float = 1.0, scale: float = 1.0,
                device="cpu") -> torch.Tensor:
    """bf16 tensor of the given shape, values bf16(fp32(N(0,std)) * scale)."""
    numel = 1
    for d in shape:
        numel *= int(d)
    v = _normal_fp32(numel, seed, tensor_id, std, scale, device)
    return v.to(torch.bfloat16).reshape(shape)


def uniform_ids(n: int, vocab: int, seed: int, tensor_id: int, device="cpu") -> torch.Tensor:
    """int32 token ids uniform in [0, vocab)."""
    k1, k2 = _keys(seed, tensor_id)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    a, _ = _hash_pair(idx, k1, k2)
    return (a % vocab).to(torch.int32)


# tensor ids: globals below 16, layer l tensor j -> 16 + 16*l + j
TID_EMBED, TID_LM_HEAD, TID_PROMPT, TID_MICRO_H, TID_MICRO_W, TID_MICRO_PRIOR = 1, 2, 3, 4, 5, 6
LAYER_TENSORS = ["attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd"]


def _layer_tid(layer: int, j: int) -> int:
    return 16 + 16 * layer + j


def gen_weights(shape: ModelShape, alpha: float, seed: int = 0, std: float = 0.02,
                device="cpu", layers: Optional[List[int]] = None) -> Dict[str, torch.Tensor]:
    """Synthetic weights in the [out_features][in_features] (row-major) convention.

    Keys: ``embed`` [V][d], ``final_norm`` [d], ``lm_head`` [V][d] (absent when tied),
    and per layer ``l{i}.{name}`` for name in LAYER_TENSORS.  W_o and W_down carry the
    residual-branch scale alpha, applied in fp32 before the bf16 rounding.  Norm gains
    are ones.
    """
    d, hd = shape.d_model, shape.head_dim
    qd, kvd = shape.n_heads * hd, shape.n_kv_heads * hd
    w: Dict[str, torch.Tensor] = {}
    w["embed"] = normal_bf16((shape.vocab, d), seed, TID_EMBED, std, device=device)
    w["final_norm"] = torch.ones(d, dtype=torch.bfloat16, device=device)
    if not shape.tied_head:
        w["lm_head"] = normal_bf16((shape.vocab, d), seed, TID_LM_HEAD, std, device=device)
    for l in (range(shape.n_layers) if layers is None else layers):
        dims = {"wq": (qd, d), "wk": (kvd, d), "wv": (kvd, d), "wo": (d, qd),
                "wg": (shape.d_ff, d), "wu": (shape.d_ff, d), "wd": (d, shape.d_ff)}
        for j, name in enumerate(LAYER_TENSORS):
            key = f"l{l}.{name}"
            if name.endswith("norm"):
                w[key] = torch.ones(d, dtype=torch.bfloat16, device=device)
            else:
                scale = alpha if name in ("wo", "wd") else 1.0
                w[key] = normal_bf16(dims[name], seed, _layer_tid(l, j), std, scale, device)
    return w


ADAPTER_TENSORS = ["g", "w1", "b1", "w2", "b2"]   # RMSNorm gain, W1 [2d][d], b1 [2d], W2 [d][2d], b2 [d]


def gen_adapters(shape: ModelShape, X: List[int], seed: int = 5, std: float = 0.02, gate: float = 0.3,
                 device="cpu") -> List[Dict[str, torch.Tensor]]:
    """Synthetic inducing adapters for the non-final depths X[0..N-2] (hidden width 2d).

    Per adapter: ``g`` RMSNorm gain (ones), ``w1`` [2d][d], ``b1`` [2d], ``w2`` [d][2d],
    ``b2`` [d] (bf16, N(0, std)) and ``alpha`` (a Python float, the scalar gate).
    """
    d = shape.d_model
    out = []
    for k in range(len(X) - 1):
        base = 4096 + 16 * k   # tensor ids of adapter k
        out.append({"g": torch.ones(d, dtype=torch.bfloat16, device=device),
                    "w1": normal_bf16((2 * d, d), seed, base + 1, std, device=device),
                    "b1": normal_bf16((2 * d,), seed, base + 2, std, device=device),
                    "w2": normal_bf16((d, 2 * d), seed, base + 3, std, device=device),
                    "b2": normal_bf16((d,), seed, base + 4, std, device=device),
                    "alpha": float(gate)})
    return out


def gen_prompts(shape: ModelShape, batch: int, prompt_len: int, seed: int = 1,
                device="cpu") -> torch.Tensor:
    """[batch][prompt_len] int32 prompt ids, uniform in [0, vocab); row b uses stream seed+b."""
    rows = [uniform_ids(prompt_len, shape.vocab, seed + b, TID_PROMPT, device) for b in range(batch)]
    return torch.stack(rows)


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bit patterns (for the oracle)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


# ----------------------------------------------------------------------------------------
# exit-head + DECS / collapse micro-benchmark inputs
# ----------------------------------------------------------------------------------------

@dataclass(frozen=True)
class ExitMicro:
    """Exit head + DECS in isolation: n_slots slot chains x depth nodes each."""
    n_slots: int = 8
    depth: int = 8
    d_model: int = 4096
    vocab: int = 128256
    seed: int = 3
    std: float = 0.02


def gen_exit_micro(m: ExitMicro, device="cpu"):
    """Hidden states [n][d] ~ N(0,1) bf16 and LM head [V][d] ~ N(0, std) bf16.

    Node order is slot-major: node = slot * depth + k, k = depth index in the slot chain.
    """
    n = m.n_slots * m.depth
    h = normal_bf16((n, m.d_model), m.seed, TID_MICRO_H, 1.0, device=device)
    w = normal_bf16((m.vocab, m.d_model), m.seed, TID_MICRO_W, m.std, device=device)
    return h, w


@dataclass(frozen=True)
class CollapseMicro:
    """KV collapse in isolation: surviving branch positions copied into the committed cache."""
    n_layers: int = 32
    n_kv_heads: int = 8
    head_dim: int = 128
    ctx: int = 4096
    n_positions: int = 6
    seed: int = 3

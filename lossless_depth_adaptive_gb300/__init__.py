"""GB300 (sm_103a) Depth Exploration Decoding: Python binding of the C ABI in include/dex.h.

This module only marshals arguments into ``_build/libdex.so``; every step of a DEX round
runs in the library's CUDA kernels and host scheduler.  Device memory and streams come
from PyTorch tensors / streams (``tensor.data_ptr()``, ``stream.cuda_stream``).

Importing does not need a GPU.  The library itself must exist (``build()`` in
``lossless_depth_adaptive_gb300.build`` or ``__graft_entry__.build()``); a missing library
raises ``DexLibraryMissing`` -- there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libdex.so")

LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")

DEX_OK, DEX_EINVAL, DEX_ENOMEM, DEX_ECUDA, DEX_ECAPACITY, DEX_ETIMEOUT, DEX_ESTATE, DEX_ENODEV, DEX_ERANGE = \
    0, -1, -2, -3, -4, -5, -6, -7, -8


class DexLibraryMissing(ImportError):
    pass


class DexError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {code} ({strerror(code)})")


class dex_model(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("d_ff", C.c_int32),
                ("vocab", C.c_int32), ("rms_eps", C.c_float), ("rope_theta", C.c_float),
                ("embed", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", C.c_void_p),
                ("layers", C.POINTER(C.c_void_p)), ("adapters", C.POINTER(C.c_void_p)),
                ("adapter_alpha", C.POINTER(C.c_float))]


class dex_decode_cfg(C.Structure):
    _fields_ = [("batch", C.c_int32), ("max_ctx", C.c_int32), ("max_new", C.c_int32),
                ("sample", C.c_int32), ("tau", C.c_float), ("seed", C.c_uint64),
                ("decs", C.c_int32), ("debug_logits", C.c_int32), ("max_branch", C.c_int32)]


class dex_stats(C.Structure):
    _fields_ = [("rounds", C.c_int64), ("commits", C.c_int64), ("nodes", C.c_int64),
                ("max_round_nodes", C.c_int64), ("layer_passes", C.c_int64),
                ("node_layers", C.c_int64), ("depth_charge", C.c_int64),
                ("kstar_hist", C.c_int64 * 16), ("weight_bytes", C.c_int64), ("kv_bytes", C.c_int64),
                ("h2d_bytes", C.c_int64), ("d2h_bytes", C.c_int64), ("kernel_launches", C.c_int64),
                ("gemm_launches", C.c_int64), ("gemm_bytes", C.c_int64), ("ms_gemm", C.c_double),
                ("ms_expand", C.c_double), ("ms_exit", C.c_double), ("ms_collapse", C.c_double),
                ("ms_host", C.c_double), ("attn_launches", C.c_int64), ("ms_attn", C.c_double)]

    def as_dict(self) -> Dict:
        d = {k: getattr(self, k) for k, _ in self._fields_}
        d["kstar_hist"] = list(self.kstar_hist)
        return d


class dex_exit_node(C.Structure):
    _fields_ = [("seq", C.c_int32), ("target_pos", C.c_int32), ("unmasked", C.c_int32),
                ("prior_off", C.c_int32), ("n_prior", C.c_int32)]


class dex_kv_geom(C.Structure):
    _fields_ = [("batch", C.c_int32), ("n_layers", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("max_ctx", C.c_int32), ("n_slots", C.c_int32)]


class dex_copy_job(C.Structure):
    _fields_ = [("seq", C.c_int32), ("slot", C.c_int32), ("pos", C.c_int32), ("n_layers", C.c_int32)]


class dex_plan_node(C.Structure):
    _fields_ = [("seq", C.c_int32), ("heap", C.c_int32), ("stage", C.c_int32), ("plen", C.c_int32),
                ("pos", C.c_int32), ("c_end", C.c_int32), ("slot", C.c_int32), ("kv_commit", C.c_int32),
                ("token", C.c_int32), ("target_pos", C.c_int32), ("unmasked", C.c_int32),
                ("n_prior", C.c_int32), ("n_tail", C.c_int32), ("prior", C.c_int32 * 16),
                ("tail", C.c_int32 * 16)]


P = C.c_void_p
I32P = C.POINTER(C.c_int32)
# name -> (restype, argtypes): every symbol of include/dex.h
SIGNATURES = {
    "dex_init": (C.c_int, [C.POINTER(dex_model), I32P, C.c_int32, C.POINTER(dex_decode_cfg), P, C.POINTER(P)]),
    "dex_prefill": (C.c_int, [P, C.c_int32, I32P, C.c_int32]),
    "dex_step": (C.c_int, [P, I32P, I32P]),
    "dex_generate": (C.c_int, [P, I32P]),
    "dex_ar_step": (C.c_int, [P, I32P, I32P]),
    "dex_ar_generate": (C.c_int, [P, I32P]),
    "dex_get_stats": (C.c_int, [P, C.POINTER(dex_stats)]),
    "dex_reset_stats": (C.c_int, [P]),
    "dex_set_timing": (C.c_int, [P, C.c_int32]),
    "dex_last_round_nodes": (C.c_int, [P, I32P, C.c_int32, I32P]),
    "dex_debug_logits": (C.c_int, [P, C.POINTER(C.c_float), C.c_int32, I32P]),
    "dex_strerror": (C.c_char_p, [C.c_int]),
    "dex_free": (None, [P]),
    "dex_selftest_stall": (C.c_int, [P, C.c_int32]),
    "dex_exit_head_decs": (C.c_int, [P, C.c_int32, C.c_int32, P, C.c_float, P, C.c_int32, P, P, C.c_int32,
                                     C.c_float, C.c_uint64, P, P, P]),
    "dex_exit_head_decs_noalloc": (C.c_int, [P, C.c_int32, C.c_int32, P, C.c_float, P, C.c_int32, P, P,
                                             C.c_int32, C.c_float, C.c_uint64, P, P, P]),
    "dex_kv_collapse": (C.c_int, [P, P, C.POINTER(dex_kv_geom), P, C.c_int32, P, P]),
    "dex_lattice_new": (C.c_int, [I32P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.POINTER(P)]),
    "dex_lattice_start": (C.c_int, [P, C.c_int32, C.c_int32, C.c_int32]),
    "dex_lattice_plan": (C.c_int, [P, C.POINTER(dex_plan_node), C.c_int32, I32P]),
    "dex_lattice_update": (C.c_int, [P, I32P, I32P, I32P, C.POINTER(dex_copy_job), C.c_int32, I32P]),
    "dex_lattice_state": (C.c_int, [P, C.c_int32, I32P, I32P, I32P]),
    "dex_lattice_free": (None, [P]),
}

_lib: Optional[C.CDLL] = None


def lib() -> C.CDLL:
    """Load libdex.so (once).  Raises DexLibraryMissing when it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise DexLibraryMissing(f"{LIB_PATH} is missing: run lossless_depth_adaptive_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def strerror(code: int) -> str:
    try:
        return lib().dex_strerror(code).decode()
    except DexLibraryMissing:
        return str(code)


def check(code: int, where: str) -> int:
    if code != DEX_OK:
        raise DexError(code, where)
    return code


def i32(values: Sequence[int]):
    return (C.c_int32 * len(values))(*values)


# ---- thin wrappers with the C names ---------------------------------------------------------

def dex_init(model: dex_model, X: Sequence[int], cfg: dex_decode_cfg, stream: int = 0) -> C.c_void_p:
    h = C.c_void_p()
    check(lib().dex_init(C.byref(model), i32(X), len(X), C.byref(cfg), C.c_void_p(stream), C.byref(h)),
          "dex_init")
    return h


def dex_prefill(h, seq: int, tokens: Sequence[int]) -> None:
    check(lib().dex_prefill(h, seq, i32(tokens), len(tokens)), "dex_prefill")


def dex_step(h, batch: int, ar: bool = False):
    out, nc = (C.c_int32 * batch)(), (C.c_int32 * batch)()
    fn = lib().dex_ar_step if ar else lib().dex_step
    check(fn(h, out, nc), "dex_ar_step" if ar else "dex_step")
    return list(out), list(nc)


def dex_ar_step(h, batch: int):
    return dex_step(h, batch, ar=True)


def dex_generate(h, batch: int, max_new: int, ar: bool = False, out=None) -> List[List[int]]:
    """Generate into ``out`` (a ctypes int32 array of batch*max_new, reused if given)."""
    if out is None:
        out = (C.c_int32 * (batch * max_new))(*([-1] * (batch * max_new)))
    fn = lib().dex_ar_generate if ar else lib().dex_generate
    check(fn(h, out), "dex_ar_generate" if ar else "dex_generate")
    return [list(out[b * max_new:(b + 1) * max_new]) for b in range(batch)]


def dex_ar_generate(h, batch: int, max_new: int) -> List[List[int]]:
    return dex_generate(h, batch, max_new, ar=True)


def dex_get_stats(h) -> Dict:
    s = dex_stats()
    check(lib().dex_get_stats(h, C.byref(s)), "dex_get_stats")
    return s.as_dict()


def dex_reset_stats(h) -> None:
    check(lib().dex_reset_stats(h), "dex_reset_stats")


def dex_set_timing(h, level: int) -> None:
    check(lib().dex_set_timing(h, level), "dex_set_timing")


def dex_last_round_nodes(h, max_rows: int = 4096) -> List[Dict]:
    buf, n = (C.c_int32 * (8 * max_rows))(), C.c_int32()
    check(lib().dex_last_round_nodes(h, buf, max_rows, C.byref(n)), "dex_last_round_nodes")
    keys = ("seq", "heap", "stage", "plen", "target_pos", "token", "n_prior", "pos")
    return [dict(zip(keys, buf[8 * k:8 * k + 8])) for k in range(n.value)]


def dex_debug_logits(h, vocab: int, max_rows: int = 512):
    import numpy as np
    out = np.zeros((max_rows, vocab), dtype=np.float32)
    n = C.c_int32()
    check(lib().dex_debug_logits(h, out.ctypes.data_as(C.POINTER(C.c_float)), max_rows, C.byref(n)),
          "dex_debug_logits")
    return out[:n.value]


def dex_free(h) -> None:
    if h:
        lib().dex_free(h)


def dex_exit_head_decs(h_ptr: int, n: int, d: int, final_norm_ptr: int, rms_eps: float, lm_head_ptr: int,
                       vocab: int, nodes_ptr: int, priors_ptr: int, sample: bool, tau: float, seed: int,
                       tokens_ptr: int, logits_ptr: int = 0, stream: int = 0) -> None:
    check(lib().dex_exit_head_decs(P(h_ptr), n, d, P(final_norm_ptr), rms_eps, P(lm_head_ptr), vocab,
                                   P(nodes_ptr), P(priors_ptr), int(sample), tau, seed, P(tokens_ptr),
                                   P(logits_ptr or None), P(stream)), "dex_exit_head_decs")


def dex_exit_head_decs_noalloc(h_ptr: int, n: int, d: int, final_norm_ptr: int, rms_eps: float,
                               lm_head_ptr: int, vocab: int, nodes_ptr: int, priors_ptr: int, sample: bool,
                               tau: float, seed: int, tokens_ptr: int, logits_ptr: int = 0, stream: int = 0) -> int:
    """Allocation-free exit head + DECS; returns the status code (raises on other errors)."""
    rc = lib().dex_exit_head_decs_noalloc(P(h_ptr), n, d, P(final_norm_ptr), rms_eps, P(lm_head_ptr), vocab,
                                          P(nodes_ptr), P(priors_ptr), int(sample), tau, seed, P(tokens_ptr),
                                          P(logits_ptr or None), P(stream))
    if rc not in (DEX_OK, DEX_ECAPACITY):
        check(rc, "dex_exit_head_decs_noalloc")
    return rc


def dex_kv_collapse(committed_ptr: int, pool_ptr: int, geom: dex_kv_geom, jobs_ptr: int, n_jobs: int,
                    stream: int = 0, rejected_ptr: int = 0) -> None:
    """rejected_ptr: device int32 that receives the number of out-of-range jobs skipped (or 0)."""
    check(lib().dex_kv_collapse(P(committed_ptr), P(pool_ptr), C.byref(geom), P(jobs_ptr), n_jobs,
                                P(rejected_ptr or None), P(stream)), "dex_kv_collapse")


# ---- model marshalling (PyTorch tensors -> dex_model) -------------------------------------------

class ModelRef:
    """Keeps the ctypes model description and the layer-pointer array alive."""

    def __init__(self, shape, weights: Dict, adapters: Optional[Sequence[Dict]] = None):
        ptrs = []
        for l in range(shape.n_layers):
            for name in LAYER_TENSORS:
                t = weights[f"l{l}.{name}"]
                assert t.is_cuda and t.is_contiguous()
                ptrs.append(t.data_ptr())
        self._layers = (C.c_void_p * len(ptrs))(*ptrs)
        head = weights["embed"] if shape.tied_head else weights["lm_head"]
        self.model = dex_model(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                               shape.d_ff, shape.vocab, shape.rms_eps, shape.rope_theta,
                               weights["embed"].data_ptr(), weights["final_norm"].data_ptr(), head.data_ptr(),
                               C.cast(self._layers, C.POINTER(C.c_void_p)))
        self.weights = weights
        self.adapters = adapters
        if adapters:
            aptrs = []
            for ad in adapters:
                for name in ("g", "w1", "b1", "w2", "b2"):
                    t = ad[name]
                    assert t.is_cuda and t.is_contiguous()
                    aptrs.append(t.data_ptr())
            self._adapters = (C.c_void_p * len(aptrs))(*aptrs)
            self._alpha = (C.c_float * len(adapters))(*[float(ad["alpha"]) for ad in adapters])
            self.model.adapters = C.cast(self._adapters, C.POINTER(C.c_void_p))
            self.model.adapter_alpha = C.cast(self._alpha, C.POINTER(C.c_float))


class Decoder:
    """A handle plus the model it references: init / prefill / step / generate / stats."""

    def __init__(self, shape, weights: Dict, X: Sequence[int], batch: int, max_ctx: int, max_new: int,
                 sample: bool = False, tau: float = 1.0, seed: int = 0, decs: bool = True,
                 debug_logits: bool = False, stream: Optional[int] = None, max_branch: int = 0,
                 adapters: Optional[Sequence[Dict]] = None):
        import torch
        self.shape, self.X, self.batch, self.max_new = shape, list(X), batch, max_new
        self.ref = ModelRef(shape, weights, adapters)
        cfg = dex_decode_cfg(batch, max_ctx, max_new, int(sample), tau, seed, int(decs), int(debug_logits),
                             int(max_branch))
        self.stream = torch.cuda.current_stream().cuda_stream if stream is None else stream
        self.h = dex_init(self.ref.model, self.X, cfg, self.stream)

    def prefill(self, seq: int, tokens: Sequence[int]) -> None:
        dex_prefill(self.h, seq, [int(t) for t in tokens])

    def step(self, ar: bool = False):
        return dex_step(self.h, self.batch, ar)

    def generate(self, ar: bool = False, out=None) -> List[List[int]]:
        return dex_generate(self.h, self.batch, self.max_new, ar, out)

    def stats(self) -> Dict:
        return dex_get_stats(self.h)

    def reset_stats(self) -> None:
        dex_reset_stats(self.h)

    def set_timing(self, level: int) -> None:
        dex_set_timing(self.h, level)

    def last_round_nodes(self) -> List[Dict]:
        return dex_last_round_nodes(self.h)

    def debug_logits(self):
        return dex_debug_logits(self.h, self.shape.vocab)

    def selftest_stall(self, limit_us: int) -> int:
        """Return code of dex_selftest_stall (DEX_ETIMEOUT when the bounded wait gave up)."""
        return lib().dex_selftest_stall(self.h, int(limit_us))

    def close(self) -> None:
        if self.h:
            dex_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Lattice:
    """Host-only lattice scheduler (the library's FSM), usable without a GPU."""

    def __init__(self, X: Sequence[int], batch: int, decs: bool = True, max_branch: int = 0):
        self.h = C.c_void_p()
        self.batch = batch
        check(lib().dex_lattice_new(i32(X), len(X), batch, int(decs), int(max_branch), C.byref(self.h)),
              "dex_lattice_new")
        self.cap = batch << (len(X) - 1)

    def start(self, seq: int, p_c: int, last_token: int) -> None:
        check(lib().dex_lattice_start(self.h, seq, p_c, last_token), "dex_lattice_start")

    def plan(self) -> List[Dict]:
        buf, n = (dex_plan_node * self.cap)(), C.c_int32()
        check(lib().dex_lattice_plan(self.h, buf, self.cap, C.byref(n)), "dex_lattice_plan")
        out = []
        for k in range(n.value):
            p = buf[k]
            d = {f: getattr(p, f) for f, _ in dex_plan_node._fields_ if f not in ("prior", "tail")}
            d["prior"] = list(p.prior[:p.n_prior])
            d["tail"] = list(p.tail[:p.n_tail])
            out.append(d)
        return out

    def update(self, tokens: Sequence[int]):
        committed, kstar = (C.c_int32 * self.batch)(), (C.c_int32 * self.batch)()
        jobs, nj = (dex_copy_job * self.batch)(), C.c_int32()
        check(lib().dex_lattice_update(self.h, i32(tokens) if tokens else None, committed, kstar, jobs,
                                       self.batch, C.byref(nj)), "dex_lattice_update")
        return list(committed), list(kstar), [(j.seq, j.slot, j.pos, j.n_layers) for j in jobs[:nj.value]]

    def state(self, seq: int):
        q, p_c, used = C.c_int32(), C.c_int32(), C.c_int32()
        check(lib().dex_lattice_state(self.h, seq, C.byref(q), C.byref(p_c), C.byref(used)), "dex_lattice_state")
        return q.value, p_c.value, used.value

    def __del__(self):
        try:
            if self.h:
                lib().dex_lattice_free(self.h)
        except Exception:
            pass

#!/usr/bin/env python
"""Benchmark: committed tokens/s and layers per committed token of DEX decoding on GB300.

Workload (default): Llama-2-7B-shaped decoder (32 layers, d 4096, 32 x 128 MHA, SwiGLU
11008, vocab 32000, seeded bf16 weights, residual scale alpha 0.05), exploration set
X = {8, 16, 24, 32}, batch 1, prompt of 512 uniform-random ids, 256 greedy tokens.

One step = one request: prefill the prompt, then DEX rounds until 256 tokens are
committed.  ``value`` is committed tokens / device time of the decode (CUDA events on
the library's stream around dex_generate; weights, prompt KV and lattice state resident
in HBM; the prefill of the next step happens outside the timed windows).  ``e2e`` is the
same request timed end to end through the C ABI with host buffers: host prompt in,
prefill, decode, host tokens out.  The weights (13.5 GB) exceed L2 (129 MB) many times
over, so no flush is needed between steps.

Multi-GPU: replicas only (one independent request stream per rank, launched with
torch.distributed.run); ``value`` = all ranks' tokens / the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle (oracle/) on the same workload and the same
decode-only unit: the prompt is prefilled once outside the timed region, and each step
decodes a bounded sample of committed tokens from that prefilled state.

Ablations (section 4.1 of the paper): ``--X 4,32`` replaces the exploration set (the
single-exit variant explores only d_0 and L), ``--no-decs`` decodes every lattice node
independently (vanilla), ``--ar`` times the library's plain autoregressive path on the same
kernels (the lossless reference every DEX stream equals).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dex_inputs as di  # noqa: E402

METRIC = "committed tokens/s (1 GB300, batch 1) and layers executed per committed token"
KV_ELEM_BYTES = 2   # bytes per element of the library's K/V caches (fp16)


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def rank_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_over_ranks(x, op, world, device):
    """max or sum of a per-rank float over the process group (identity at world 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def replica_throughput(tokens_per_rank, seconds_per_rank, world, device):
    """Whole-job committed tokens/s of independent replicas: all ranks' tokens over the
    slowest rank's time."""
    return (reduce_over_ranks(tokens_per_rank, "sum", world, device) /
            reduce_over_ranks(seconds_per_rank, "max", world, device))


def _gemm_traffic_ratio():
    """DRAM bytes per algorithmic byte of gemm_tc_kernel from the committed ncu summary, if
    that summary was taken on the current gemm.cu (else None: the counters are stale)."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "gemm_tc_kernel_grouped_l4.md")
    src = os.path.join(ROOT, "lossless_depth_adaptive_gb300", "csrc", "gemm.cu")
    try:
        text = open(prof).read()
        ratio = float(text.split("dram_over_algorithmic:")[1].split()[0])
        sha = text.split("gemm_cu_sha256_16:")[1].split()[0]
    except (OSError, IndexError, ValueError):
        return None
    with open(src, "rb") as f:
        return ratio if hashlib.sha256(f.read()).hexdigest()[:16] == sha else None


MODEL_NAMES = {di.LLAMA7B: "llama2-7b-shaped", di.QWEN8B: "qwen3-8b-shaped", di.TINY: "tiny"}


def prefill_flop(shape, batch, positions):
    """FLOP of prefilling `positions` prompt positions of `batch` sequences: every linear
    layer at 2 FLOP per weight and position (QKV, O, gate, up, down), plus causal attention
    at 4 * head_dim FLOP per (query head, query, visible key) pair -- QK^T and PV, each
    query seeing itself and every earlier position."""
    qd, kvd = shape.n_heads * shape.head_dim, shape.n_kv_heads * shape.head_dim
    layer_params = (qd + 2 * kvd) * shape.d_model + qd * shape.d_model + 3 * shape.d_ff * shape.d_model
    pairs = positions * (positions + 1) / 2
    return batch * shape.n_layers * (2.0 * layer_params * positions + 4.0 * qd * pairs)


def _weight_gb(shape):
    qd, kvd = shape.n_heads * shape.head_dim, shape.n_kv_heads * shape.head_dim
    per_layer = (qd + 2 * kvd) * shape.d_model + qd * shape.d_model + 3 * shape.d_ff * shape.d_model
    return (shape.n_layers * per_layer + shape.vocab * shape.d_model) * 2 / 1e9


def _workload(args):
    over = {}
    if args.tokens:
        over["max_new"] = args.tokens
    if getattr(args, "alpha", None) is not None:
        over["alpha"] = args.alpha
    if getattr(args, "X", None):
        over["X"] = [int(x) for x in args.X.split(",")]
    if getattr(args, "no_decs", False):
        over["decs"] = False
    return di.workload(args.workload, **over)


def _config(args, wl, world, B):
    """The workload description both arms print (same keys, so the lines compare)."""
    return {"workload": wl.name, "model": MODEL_NAMES.get(wl.shape, "decoder"), "X": wl.X, "alpha": wl.alpha,
            "global_batch": world * B, "prompt_len": wl.prompt_len, "new_tokens": wl.max_new,
            "decode": "sample" if wl.sample else "greedy", "decs": bool(wl.decs),
            "path": "ar" if getattr(args, "ar", False) else "dex", "parallelism": f"replicas{world}",
            "max_branch": args.max_branch, "adapters": _adapter_cfg(args, wl),
            "l2": f"weights {_weight_gb(wl.shape):.1f} GB streamed per round >> 129 MB L2; no flush"}


def run_gpu(args):
    import torch
    import lossless_depth_adaptive_gb300 as dexlib

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    wl = _workload(args)
    shape = wl.shape
    w = di.gen_weights(shape, wl.alpha, seed=wl.weight_seed, device="cuda")
    B = wl.batch   # independent sequences decoded together (one request each)
    prompts = di.gen_prompts(shape, B, wl.prompt_len, seed=wl.prompt_seed + 1000 * rank).tolist()
    prompt = prompts[0]
    T = wl.max_new
    max_ctx = wl.prompt_len + T + len(wl.X) + 8
    ads = _adapters(args, wl, "cuda")
    dec = dexlib.Decoder(shape, w, wl.X, batch=B, max_ctx=max_ctx, max_new=T, sample=wl.sample, tau=wl.tau,
                         seed=wl.gumbel_seed, decs=wl.decs, max_branch=args.max_branch, adapters=ads)
    st = torch.cuda.current_stream()
    import ctypes as C
    out_host = (C.c_int32 * (B * T))()

    def prefill_all():
        for b in range(B):
            dec.prefill(b, prompts[b])

    dev = torch.device("cuda", local)

    def barrier():
        torch.cuda.synchronize()
        rank_barrier(world)

    def max_over_ranks(x):
        return reduce_over_ranks(x, "max", world, dev)

    # warm-up requests
    AR = bool(args.ar)
    for _ in range(args.warmup):
        prefill_all()
        dec.generate(ar=AR, out=out_host)
    # ---- device-timed decode (value) ----
    dec.reset_stats()
    barrier()
    ms = 0.0
    tokens_ref = None
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            prefill_all()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            toks = dec.generate(ar=AR, out=out_host)
            e1.record(st)
            e1.synchronize()
            ms += e0.elapsed_time(e1)
            if tokens_ref is None:
                tokens_ref = toks
            assert toks == tokens_ref, "decode is not deterministic across requests"
    barrier()
    stats = dec.stats()
    launches = stats["kernel_launches"]
    # ---- prefill alone (support path, not the timed metric): device time of the prompts ----
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record(st)
    prefill_all()
    pe1.record(st)
    pe1.synchronize()
    prefill_ms = pe0.elapsed_time(pe1)
    prefill_tok = B * (wl.prompt_len - 1)
    pf_flop = prefill_flop(shape, B, wl.prompt_len - 1)
    value = replica_throughput(args.steps * B * T, ms / 1000.0, world, dev)
    ms = max_over_ranks(ms)
    ms_per_step = ms / args.steps
    # ---- end to end through the C ABI with host buffers (e2e) ----
    dec.reset_stats()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        prefill_all()                        # host prompts -> device inside
        dec.generate(ar=AR, out=out_host)    # tokens -> host inside
    barrier()
    e2e_value = replica_throughput(args.steps * B * T, time.perf_counter() - t0, world, dev)
    st_e2e = dec.stats()
    e2e = {"value": e2e_value, "unit": "committed tokens/s",
           "h2d_bytes_per_step": int(st_e2e["h2d_bytes"] / args.steps),
           "d2h_bytes_per_step": int(st_e2e["d2h_bytes"] / args.steps)}
    # ---- one instrumented request: per-GEMM events and phase split ----
    dec.set_timing(2)
    dec.reset_stats()
    prefill_all()
    dec.reset_stats()
    dec.generate(ar=AR, out=out_host)
    inst = dec.stats()
    dec.set_timing(0)
    dec.close()
    hbm, bf16, src = _peaks()
    achieved = inst["gemm_bytes"] / (inst["ms_gemm"] / 1000.0) / 1e9 if inst["ms_gemm"] > 0 else None
    ratio = _gemm_traffic_ratio()
    bytes_per_launch = inst["gemm_bytes"] / max(1, inst["gemm_launches"])
    commits = stats["commits"]
    # algorithmic bytes: every live layer's weights once per round, the LM head once per
    # round, the KV entries attention must read counted at 2 bytes per element (the cache's
    # own element size is reported beside it)
    kv_algo = stats["kv_bytes"] * 2 // KV_ELEM_BYTES
    algo_bytes = stats["weight_bytes"] + kv_algo
    step_roof = {"algorithmic_bytes_per_step": int(algo_bytes / args.steps),
                 "kv_bytes_per_step": int(kv_algo / args.steps), "kv_cache_elem_bytes": KV_ELEM_BYTES,
                 "roofline_ms_per_step": algo_bytes / args.steps / (hbm * 1e9) * 1e3,
                 "frac": (algo_bytes / (hbm * 1e9)) / (ms / 1e3) if ms > 0 else None,
                 "frac_of": f"measured {hbm:.0f} GB/s ({src})",
                 "frac_8tbs": (algo_bytes / 8e12) / (ms / 1e3) if ms > 0 else None}
    layers = {"depth_charge_per_token": stats["depth_charge"] / commits,
              "layer_passes_per_token": stats["layer_passes"] / commits,
              "node_layers_per_token": stats["node_layers"] / commits,
              "rounds_per_token": stats["rounds"] / commits,
              "nodes_per_round": stats["nodes"] / stats["rounds"],
              "kstar_hist": stats["kstar_hist"][:len(wl.X)],
              # depth-side speedup (Eq. 12): L T / sum_t W(t), W(t) the depth charged to token t
              "depth_side_speedup": shape.n_layers * commits / stats["depth_charge"] if stats["depth_charge"] else None}
    phases = {k: inst[k] / inst["rounds"] for k in ("ms_expand", "ms_exit", "ms_collapse", "ms_host")}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "committed tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded weights and uniform-random prompt ids)",
        "config": _config(args, wl, world, B),
        "layers_per_token": {k: (round(v, 3) if isinstance(v, float) else v) for k, v in layers.items()},
        "step_roofline": step_roof,
        "phase_ms_per_round": {k: round(v, 4) for k, v in phases.items()},
        "attention": {"launches": inst["attn_launches"],
                      "us_per_launch": round(inst["ms_attn"] * 1e3 / max(1, inst["attn_launches"]), 2),
                      "kv_gbs": round(inst["kv_bytes"] / (inst["ms_attn"] / 1e3) / 1e9, 1) if inst["ms_attn"] else None,
                      "share_of_request": round(inst["ms_attn"] / ms_per_step, 4) if ms_per_step else None,
                      "note": "CUDA events around each launch in one instrumented request (no launch overlap)"},
        "roofline": {"bound": "hbm", "kernel": "gemm_tc_kernel (all linear layers, one instrumented request)",
                     "achieved": round(achieved, 1) if achieved else None, "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4) if achieved else None, "peak_source": src,
                     "frac_8tbs": round(achieved / 8000.0, 4) if achieved else None,
                     "traffic": int(ratio * bytes_per_launch) if ratio else None,
                     "traffic_source": "ncu dram bytes / algorithmic bytes (profiles/gemm_tc_kernel_grouped_l4.md)"
                                       " x this run's algorithmic bytes per launch" if ratio else None,
                     "launches": inst["gemm_launches"], "bytes_per_launch": int(bytes_per_launch),
                     "ms_per_launch": inst["ms_gemm"] / max(1, inst["gemm_launches"])},
        "e2e": e2e,
        "prefill": {"tokens": prefill_tok, "ms": round(prefill_ms, 2),
                    "tokens_per_s": round(prefill_tok / (prefill_ms / 1e3), 1) if prefill_ms > 0 else None,
                    "tflops": round(pf_flop / (prefill_ms / 1e3) / 1e12, 1) if prefill_ms > 0 else None,
                    "frac_of_bf16_peak": round(pf_flop / (prefill_ms / 1e3) / 1e12 / bf16, 4)
                    if prefill_ms > 0 else None,
                    "note": "support path (not the metric): prompt positions 0..P-2 of every sequence, "
                            "linear layers at 2 FLOP per weight and token plus causal attention"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args, wl, w, prompt, ads)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_micro(args):
    """Exit head + DECS and the KV collapse in isolation (the kernel micro-benchmark shapes):
    64 lattice nodes (8 slot chains x 8 depths, 0-7 masked priors each, sampled with shared
    Gumbel rows) against a 128256 x 4096 bf16 LM head; 6 surviving branch positions copied
    into a 32-layer x 8-KV-head x 128 bf16 cache at context 4096."""
    import torch
    import lossless_depth_adaptive_gb300 as dexlib
    torch.cuda.set_device(_dist()[2])
    m = di.ExitMicro()
    h, w = di.gen_exit_micro(m, device="cuda")
    n, d, V = m.n_slots * m.depth, m.d_model, m.vocab
    g = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    ids = di.uniform_ids(n * m.depth, V, m.seed, 7).tolist()
    nodes, priors = [], []
    for sl in range(m.n_slots):
        for k in range(m.depth):
            unmasked = 1 if k == m.depth - 1 else 0
            pr = [] if unmasked else ids[(sl * m.depth + k) * m.depth:][:k]
            nodes.append((sl, 1000 + sl, unmasked, len(priors), len(pr)))
            priors += pr
    nodes_t = torch.tensor(nodes, dtype=torch.int32, device="cuda")
    priors_t = torch.tensor(priors + [0], dtype=torch.int32, device="cuda")
    tokens = torch.empty(n, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()

    def exit_call():
        dexlib.dex_exit_head_decs(h.data_ptr(), n, d, g.data_ptr(), 1e-5, w.data_ptr(), V, nodes_t.data_ptr(),
                                  priors_t.data_ptr(), 1, 0.7, 2, tokens.data_ptr(), 0, st.cuda_stream)

    def exit_call_noalloc():
        dexlib.dex_exit_head_decs_noalloc(h.data_ptr(), n, d, g.data_ptr(), 1e-5, w.data_ptr(), V,
                                          nodes_t.data_ptr(), priors_t.data_ptr(), 1, 0.7, 2, tokens.data_ptr(),
                                          0, st.cuda_stream)

    cm = di.CollapseMicro()
    S = 8
    committed = torch.zeros((1, cm.n_layers, 2, cm.n_kv_heads, cm.ctx, cm.head_dim), dtype=torch.bfloat16,
                            device="cuda")
    pool = torch.ones((1, S, cm.n_layers, 2, cm.n_kv_heads, cm.head_dim), dtype=torch.bfloat16, device="cuda")
    jobs = torch.tensor([(0, j, cm.ctx - 1 - 7 * j, cm.n_layers) for j in range(cm.n_positions)], dtype=torch.int32,
                        device="cuda")
    geom = dexlib.dex_kv_geom(1, cm.n_layers, cm.n_kv_heads, cm.head_dim, cm.ctx, S)

    def collapse_call():
        dexlib.dex_kv_collapse(committed.data_ptr(), pool.data_ptr(), geom, jobs.data_ptr(), cm.n_positions,
                               st.cuda_stream)

    def timed(fn, reps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            fn()
        e1.record(st)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3   # us

    hbm, _, src = _peaks()
    with ClockSampler(_dist()[2]) as clk:
        t_exit = timed(exit_call, max(10, args.steps * 10))
        t_exit_na = timed(exit_call_noalloc, max(10, args.steps * 10))
        t_col = timed(collapse_call, max(10, args.steps * 10))
    exit_bytes = V * d * 2 + n * d * 2 + len(priors) * 4
    col_bytes = 2 * cm.n_positions * cm.n_layers * 2 * cm.n_kv_heads * cm.head_dim * 2
    line = {"metric": "exit head + DECS (64 nodes, LM head 128256 x 4096 bf16) and KV collapse "
                      "(6 positions, 32 layers x 8 KV heads x 128, context 4096), isolated",
            "value": round(exit_bytes / (t_exit * 1e-6) / 1e9, 1), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": "micro", "nodes": n, "vocab": V, "d_model": d,
                                            "sample": True, "collapse_positions": cm.n_positions},
            "exit_head": {"us_per_call": round(t_exit, 2), "bytes": exit_bytes,
                          "frac_of_hbm": round(exit_bytes / (t_exit * 1e-6) / 1e9 / hbm, 4), "peak_source": src,
                          "grid": "2 CTAs per SM"},
            "exit_head_noalloc": {"us_per_call": round(t_exit_na, 2),
                                  "frac_of_hbm": round(exit_bytes / (t_exit_na * 1e-6) / 1e9 / hbm, 4),
                                  "grid": "1 CTA per SM (fixed 32 MiB scratch)"},
            "collapse": {"us_per_call": round(t_col, 2), "bytes_moved": col_bytes,
                         "gbs": round(col_bytes / (t_col * 1e-6) / 1e9, 2)},
            "clocks": clk.summary()}
    print(json.dumps(line))


def _oracle_for(wl, w_gpu):
    from oracle.model import OracleModel
    bits = {k: di.bf16_bits(v) for k, v in w_gpu.items()}
    return OracleModel(wl.shape, bits, keep_widened=True)


def _adapters(args, wl, device):
    """Seeded inducing adapters at the non-final exits when --adapters GATE is given."""
    if args.adapters is None:
        return None
    return di.gen_adapters(wl.shape, wl.X, gate=args.adapters, device=device)


def _adapter_cfg(args, wl):
    if args.adapters is None:
        return None
    return {"gate": args.adapters, "hidden": 2 * wl.shape.d_model, "count": len(wl.X) - 1, "weights": "seeded"}


def _oracle_adapters(ads):
    if ads is None:
        return None
    from oracle.model import widen_bf16
    return [{k: (v if k == "alpha" else widen_bf16(di.bf16_bits(v))) for k, v in a.items()} for a in ads]


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() in ("Model name", "Model"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


class _OneCore:
    """Run numpy's BLAS on one thread and the process on one core for the block (the
    OpenBLAS thread count is set through its own C entry point, found among the loaded
    libraries); ``ok`` is False when no BLAS control was found."""

    def __enter__(self):
        import ctypes
        self.ok, self.restore, self.set_fn = False, None, None
        try:
            maps = open("/proc/self/maps").read().split("\n")
        except OSError:
            maps = []
        libs = sorted({ln.split()[-1] for ln in maps if "openblas" in ln.lower() and ln.split()[-1].startswith("/")})
        for path in libs:
            try:
                h = ctypes.CDLL(path, mode=getattr(os, "RTLD_NOLOAD", 4) | ctypes.RTLD_GLOBAL)
            except OSError:
                continue
            for stem in ("scipy_openblas", "openblas"):
                for suf in ("64_", ""):
                    get = getattr(h, f"{stem}_get_num_threads{suf}", None)
                    put = getattr(h, f"{stem}_set_num_threads{suf}", None)
                    if get is not None and put is not None:
                        self.restore, self.set_fn = get(), put
                        put(1)
                        self.ok = True
                        break
                if self.ok:
                    break
            if self.ok:
                break
        self.aff = os.sched_getaffinity(0)
        os.sched_setaffinity(0, {min(self.aff)})
        return self

    def __exit__(self, *exc):
        os.sched_setaffinity(0, self.aff)
        if self.set_fn is not None:
            self.set_fn(self.restore)


CPU_SAMPLE_TOKENS = {"tiny": 16, "llama7b_x4": 2, "llama7b_x8_sample": 1, "qwen8b_x4_b8": 1}


def _oracle_decode(args, wl, m, prompt, n_tokens, cache, ads_wide):
    """Decode n_tokens committed tokens of the workload's path with the oracle, from a
    prefilled cache; returns (tokens, rounds)."""
    from oracle import dex as odex
    rule = odex.Rule(sample=wl.sample, tau=wl.tau, seed=wl.gumbel_seed)
    if getattr(args, "ar", False):
        r = odex.ar_generate(m, prompt, n_tokens, rule=rule, cache=cache)
        return len(r.tokens), len(r.tokens)
    r = odex.dex_generate(m, prompt, wl.X, n_tokens, rule=rule, use_decs=wl.decs, max_branch=args.max_branch,
                          adapters=ads_wide, cache=cache)
    return len(r.tokens), r.rounds


def cpu_baseline(args, wl, w_gpu, prompt, ads=None):
    """Time the oracle on a bounded sample of the same decode the GPU line measures: the
    prompt is prefilled once (timed on its own), then committed tokens are decoded from that
    state on all host cores and, for one token, on one core."""
    from oracle import dex as odex
    m = _oracle_for(wl, w_gpu)
    wide = _oracle_adapters(ads)
    n = CPU_SAMPLE_TOKENS.get(wl.name, 1)
    cap = len(prompt) + n + len(wl.X) + 2
    t0 = time.perf_counter()
    cache = odex.prefill(m, prompt, cap)
    prefill_s = time.perf_counter() - t0
    t0 = time.perf_counter()
    toks, rounds = _oracle_decode(args, wl, m, prompt, n, cache, wide)
    dt = time.perf_counter() - t0
    one = None
    with _OneCore() as oc:
        t1 = time.perf_counter()
        toks1, rounds1 = _oracle_decode(args, wl, m, prompt, 1, cache, wide)
        dt1 = time.perf_counter() - t1
        if oc.ok:
            one = {"value": round(toks1 / dt1, 6), "cores": 1, "seconds": round(dt1, 2),
                   "ms_per_round": round(dt1 / rounds1 * 1e3, 1)}
    return {"value": round(toks / dt, 6), "unit": "committed tokens/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "seconds": round(dt, 2), "ms_per_round": round(dt / rounds * 1e3, 1),
            "prefill_s": round(prefill_s, 2), "prefill_positions": len(prompt) - 1, "one_core": one,
            "cpu_model": _cpu_model(),
            "sample": f"fp64 oracle: {toks} committed token(s) ({rounds} rounds) of the {wl.name} workload, "
                      f"decoded from the prefilled prompt (prefill timed separately); one sequence"}


def run_reference(args):
    """The oracle as the reference arm, on rank 0 only: the same workload, unit and config
    keys as the library's line.  Setup (weights, the fp64 model, the prompt's prefill) is
    outside the timed region; each step decodes a bounded sample of committed tokens from
    the prefilled state, like the library's decode-only ``value``."""
    rank, world, local = _dist()
    if rank != 0:
        return
    import torch
    wl = _workload(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = di.gen_weights(wl.shape, wl.alpha, seed=wl.weight_seed, device=dev)
    prompt = di.gen_prompts(wl.shape, wl.batch, wl.prompt_len, seed=wl.prompt_seed)[0].tolist()
    from oracle import dex as odex
    m = _oracle_for(wl, w)
    del w
    wide = _oracle_adapters(_adapters(args, wl, "cpu"))
    n = CPU_SAMPLE_TOKENS.get(wl.name, 1)
    t0 = time.perf_counter()
    cache = odex.prefill(m, prompt, len(prompt) + n + len(wl.X) + 2)
    prefill_s = time.perf_counter() - t0
    for _ in range(args.warmup):
        _oracle_decode(args, wl, m, prompt, n, cache, wide)
    t0 = time.perf_counter()
    toks = rounds = 0
    for _ in range(args.steps):
        a, b = _oracle_decode(args, wl, m, prompt, n, cache, wide)
        toks += a
        rounds += b
    dt = time.perf_counter() - t0
    v = toks / dt
    cores = len(os.sched_getaffinity(0))
    sample = (f"fp64 oracle: per step, {n} committed token(s) of one sequence decoded from the prefilled "
              f"{wl.prompt_len}-token prompt ({rounds / args.steps:.1f} rounds); prefill {prefill_s:.1f} s, untimed")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "committed tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded weights and uniform-random prompt ids)",
        "config": _config(args, wl, world, wl.batch),
        "cpu_baseline": {"value": round(v, 6), "unit": "committed tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": _cpu_model(), "prefill_s": round(prefill_s, 2)},
        "e2e": {"value": round(v, 6), "unit": "committed tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["dex", "reference"], default="dex")
    ap.add_argument("--workload", default="llama7b_x4", choices=sorted(di.WORKLOADS) + ["micro"],
                    help="micro: exit head + DECS and KV collapse in isolation")
    ap.add_argument("--tokens", type=int, default=0, help="override the new-token count")
    ap.add_argument("--alpha", type=float, default=None,
                    help="override the residual-branch scale (sets how often shallow exits agree)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--max-branch", type=int, default=0,
                    help="sparse lattice: nodes speculate at most this many tokens ahead (0: full lattice)")
    ap.add_argument("--adapters", type=float, default=None, metavar="GATE",
                    help="seeded inducing adapters (hidden width 2d) at the non-final exits, scalar gate GATE")
    ap.add_argument("--X", default=None, help="exploration set override, e.g. 4,32 (single-exit variant)")
    ap.add_argument("--no-decs", action="store_true", help="vanilla lattice: no depth-coupled masking")
    ap.add_argument("--ar", action="store_true", help="time the plain autoregressive path on the same kernels")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "dex":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "micro":
        run_micro(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

"""Run one DEX request inside a profiler window (for ncu --profile-from-start off).

    python -m lossless_depth_adaptive_gb300.profile_case --workload llama7b_x4 --tokens 8
    python -m lossless_depth_adaptive_gb300.profile_case --workload llama7b_x4 --layers 4 --tokens 2
    python -m lossless_depth_adaptive_gb300.profile_case --tokens 8 --adapters 0.001
    python -m lossless_depth_adaptive_gb300.profile_case --layers 4 --prefill

Builds the workload's seeded weights (optionally only the first ``--layers`` layers, with
the exploration set rescaled to the same number of stages), prefills the prompt, runs
``--warmup`` untimed requests, then opens the CUDA profiler window for exactly one
request's decode (``--tokens`` committed tokens) and closes it; with ``--prefill`` the
window holds the prompts' prefill instead.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    import dex_inputs as di
    import lossless_depth_adaptive_gb300 as dexlib

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama7b_x4", choices=sorted(di.WORKLOADS))
    ap.add_argument("--layers", type=int, default=0, help="keep only the first n layers")
    ap.add_argument("--tokens", type=int, default=8)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--ar", action="store_true", help="profile plain autoregressive rounds")
    ap.add_argument("--max-branch", type=int, default=0, help="sparse lattice speculation cap (0: full lattice)")
    ap.add_argument("--adapters", type=float, default=None, metavar="GATE",
                    help="seeded inducing adapters at the non-final exits with scalar gate GATE")
    ap.add_argument("--timeline", action="store_true",
                    help="record per-CTA GEMM clock records of the profiled request (needs DEX_TIMELINE=<file>)")
    ap.add_argument("--prefill", action="store_true", help="profile the prompts' prefill instead of a decode")
    a = ap.parse_args()
    wl = di.workload(a.workload)
    shape, X = wl.shape, list(wl.X)
    if a.layers:
        N = len(X)
        assert a.layers % N == 0, "--layers must be a multiple of the number of stages"
        shape = di.ModelShape(**{**shape.__dict__, "n_layers": a.layers})
        X = [a.layers // N * (k + 1) for k in range(N)]
    w = di.gen_weights(shape, wl.alpha, seed=wl.weight_seed, device="cuda")
    prompts = di.gen_prompts(shape, wl.batch, wl.prompt_len, seed=wl.prompt_seed).tolist()
    ads = None if a.adapters is None else di.gen_adapters(shape, X, gate=a.adapters, device="cuda")
    dec = dexlib.Decoder(shape, w, X, batch=wl.batch, max_ctx=wl.prompt_len + a.tokens + len(X) + 8,
                         max_new=a.tokens, sample=wl.sample, tau=wl.tau, seed=wl.gumbel_seed, decs=wl.decs,
                         max_branch=a.max_branch, adapters=ads)

    def prefill_all():
        for b, p in enumerate(prompts):
            dec.prefill(b, p)

    for _ in range(a.warmup):
        prefill_all()
        dec.generate(ar=a.ar)
    if a.prefill:
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.profiler.start()
        e0.record()
        prefill_all()
        e1.record()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        n = sum(len(p) - 1 for p in prompts)
        ms = e0.elapsed_time(e1)
        print(f"profiled prefill of {n} positions, layers {shape.n_layers}: {ms:.2f} ms, "
              f"{n / ms * 1e3:.0f} positions/s")
        dec.close()
        return
    prefill_all()
    torch.cuda.synchronize()
    if a.timeline:
        dec.set_timing(3)
    torch.cuda.profiler.start()
    toks = dec.generate(ar=a.ar)[0]
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    dec.set_timing(0)
    st = dec.stats()
    dec.close()
    print(f"profiled {a.tokens} tokens ({'AR' if a.ar else 'DEX'}), layers {shape.n_layers}, X {X}: "
          f"{toks[:8]}..., kernel launches so far {st['kernel_launches']}")


if __name__ == "__main__":
    main()

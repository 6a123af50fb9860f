"""Helpers shared by the GPU tests (not collected: no test_ prefix)."""
import numpy as np
import torch

import dex_inputs as di


def require_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import lossless_depth_adaptive_gb300 as dexlib
    try:
        dexlib.lib()
    except dexlib.DexLibraryMissing:
        from lossless_depth_adaptive_gb300 import build
        build.build()
    return dexlib


def oracle_model(shape, w_gpu, keep_widened=True):
    from oracle.model import OracleModel
    return OracleModel(shape, {k: di.bf16_bits(v) for k, v in w_gpu.items()}, keep_widened=keep_widened)


def check_logits_and_tokens(gpu_logits, gpu_tokens, ref, tol=5e-2, margin=0.1, scores=None):
    """Max-abs logits error <= tol; tokens equal wherever the oracle's decision margin > margin."""
    errs, checked = [], 0
    for t, y in enumerate(gpu_tokens):
        ref_z = ref.logits[t]
        errs.append(float(np.max(np.abs(np.asarray(gpu_logits[t], np.float64) - ref_z))))
        if ref.margins[t] > margin:
            s = ref_z if scores is None else scores[t]
            assert y == int(np.argmax(s)), f"token {t}: GPU {y}, oracle {int(np.argmax(s))} (margin {ref.margins[t]})"
            checked += 1
    assert max(errs) <= tol, f"logits max-abs error {max(errs)} > {tol}"
    return max(errs), checked

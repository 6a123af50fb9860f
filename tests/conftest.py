"""Shared fixtures.  Tests marked ``gpu`` need a GB300 (sm_103a) and the built library."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running full-size check")


def golden_lines(name):
    """Non-comment, non-empty lines of a golden fixture."""
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


_MODEL_CACHE = {}


def tiny_model(alpha=0.1, tied=True, n_layers=8, seed=0):
    """Tiny-shaped oracle model (cached): the 8-layer d=256 decoder and its variants."""
    import dex_inputs as di
    from oracle.model import OracleModel
    key = (alpha, tied, n_layers, seed)
    if key not in _MODEL_CACHE:
        shape = di.ModelShape(**{**di.TINY.__dict__, "tied_head": tied, "n_layers": n_layers})
        w = di.gen_weights(shape, alpha, seed=seed)
        bits = {k: di.bf16_bits(v) for k, v in w.items()}
        _MODEL_CACHE[key] = (shape, w, OracleModel(shape, bits))
    return _MODEL_CACHE[key]

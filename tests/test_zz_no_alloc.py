"""The allocation-free exit head + DECS entry point against the fp64 exit head and the
allocating entry point.

dex_exit_head_decs_noalloc exists for callers that must not allocate device memory while
they run (code under someone else's stream capture or allocator, or with a memory budget
fixed at start-up).  It takes its scratch from a fixed device array shared by all calls,
so this test makes two calls in a row -- a split-K shape (arrival counters that must be
cleared) followed by a different, unsplit shape -- and checks each against the fp64 exit
head RMSNorm(h) W^T and DECS on it (the tolerance of the kernel tests), and against
dex_exit_head_decs (logits within 2e-3, tokens equal wherever the decision margin exceeds
0.1).  It checks that repeated calls leave the device's free memory unchanged, and that a
call needing more scratch than the fixed array is refused without running.  The file name
makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

from gpu_util import require_gpu
from oracle import dex as odex

pytestmark = pytest.mark.gpu


def _inputs(n_slots, depth, d, V, std):
    from test_gpu_kernels import exit_case_inputs
    h, w, z, nodes, priors = exit_case_inputs(n_slots, depth, d, V, std=std)
    nodes_t = torch.tensor(nodes, dtype=torch.int32, device="cuda")
    priors_t = torch.tensor(priors + [0], dtype=torch.int32, device="cuda")
    return h, w, z, nodes, priors, nodes_t, priors_t, len(nodes)


def _call(fn, h, w, nodes_t, priors_t, n, d, V, sample):
    dexlib = require_gpu()
    g = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    tokens = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    logits = torch.full((n, V), float("nan"), dtype=torch.float32, device="cuda")
    rc = getattr(dexlib, fn)(h.data_ptr(), n, d, g.data_ptr(), 1e-5, w.data_ptr(), V, nodes_t.data_ptr(),
                             priors_t.data_ptr(), sample, 0.7, 77, tokens.data_ptr(), logits.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc, tokens.cpu().numpy(), logits.cpu().numpy()


def test_noalloc_matches_allocating_entry_point_on_consecutive_calls():
    dexlib = require_gpu()
    cases = [(4, 5, 2048, 2048, 0.02, True),     # split-K: counters in the shared scratch
             (3, 4, 256, 1000, 0.2, False)]      # single split, ragged vocabulary tile
    from test_gpu_kernels import check_exit_tokens
    for n_slots, depth, d, V, std, sample in cases:
        h, w, z, nodes_l, priors_l, nodes_t, priors_t, n = _inputs(n_slots, depth, d, V, std)
        _, tok_ref, lg_ref = _call("dex_exit_head_decs", h, w, nodes_t, priors_t, n, d, V, sample)
        rc, tok, lg = _call("dex_exit_head_decs_noalloc", h, w, nodes_t, priors_t, n, d, V, sample)
        assert rc == dexlib.DEX_OK
        assert np.isfinite(lg).all()
        rule = odex.Rule(sample=sample, tau=0.7, seed=77)
        # against the fp64 exit head and DECS on its logits (the kernel tests' tolerance)
        err = float(np.max(np.abs(lg.astype(np.float64) - z)))
        assert err < 2e-3 * max(1.0, float(np.abs(z).max()) / 8), f"exit logits max-abs error {err}"
        assert check_exit_tokens(tok.tolist(), z, nodes_l, priors_l, rule) >= n // 2
        # against the allocating entry point
        assert float(np.max(np.abs(lg.astype(np.float64) - lg_ref))) <= 2e-3
        nodes = nodes_t.cpu().tolist()
        priors = priors_t.cpu().tolist()
        checked = 0
        for i, (s, pos, unm, off, cnt) in enumerate(nodes):
            zr = lg_ref[i].astype(np.float64)
            for v in priors[off:off + cnt]:
                zr[v] = -np.inf
            if odex.margin(odex.decision_scores(zr, rule, s, pos)) > 0.1:
                assert tok[i] == tok_ref[i]
                checked += 1
        assert checked > 0


def test_noalloc_calls_leave_device_memory_unchanged():
    """The point of the entry point: after the first call on the device (which looks up the
    fixed array's address), further calls take no device memory."""
    dexlib = require_gpu()
    h, w, z, nodes_l, priors_l, nodes_t, priors_t, n = _inputs(4, 5, 2048, 2048, 0.02)
    d, V = 2048, 2048
    g = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    tokens = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream

    def call():
        return dexlib.dex_exit_head_decs_noalloc(h.data_ptr(), n, d, g.data_ptr(), 1e-5, w.data_ptr(), V,
                                                 nodes_t.data_ptr(), priors_t.data_ptr(), 1, 0.7, 77,
                                                 tokens.data_ptr(), 0, st)

    assert call() == dexlib.DEX_OK
    first = tokens.clone()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch_alloc0 = torch.cuda.memory_allocated()
    for _ in range(4):
        assert call() == dexlib.DEX_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
    assert torch.cuda.memory_allocated() == torch_alloc0
    assert torch.equal(tokens, first)


def test_noalloc_refuses_oversized_calls():
    dexlib = require_gpu()
    # 256 nodes against a 8192 x 4096 head needs 8-way split-K partials of 64 MiB
    n, d, V = 256, 4096, 8192
    h = torch.zeros((n, d), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((V, d), dtype=torch.bfloat16, device="cuda")
    nodes_t = torch.zeros((n, 5), dtype=torch.int32, device="cuda")
    priors_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc, tok, _ = _call("dex_exit_head_decs_noalloc", h, w, nodes_t, priors_t, n, d, V, False)
    assert rc == dexlib.DEX_ECAPACITY
    assert (tok == -1).all()          # nothing ran

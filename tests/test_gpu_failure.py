"""Failure paths of the C ABI, produced without faulting or hanging the GPU.

* A bounded device wait that gives up: ``dex_selftest_stall`` runs the library's bounded
  mbarrier wait against a barrier nothing completes, with a 1 ms limit.  The call must
  return DEX_ETIMEOUT through the same device flag and host check as a decode round, and
  the handle must stay usable (a decode afterwards equals a fresh handle's) and freeable.
* An allocation failure inside ``dex_init``, injected on the host (DEX_FAIL_ALLOC_AT=k
  makes the k-th allocation report failure): the call returns DEX_ENOMEM, and the device's
  free memory is back where it was (nothing leaked).
"""
import os

import pytest
import torch

import dex_inputs as di
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu

SHAPE = di.ModelShape(**{**di.TINY.__dict__, "tied_head": False})
X = [2, 4, 6, 8]


def _decode(dexlib, w, prompt, T, dec=None):
    own = dec is None
    if own:
        dec = dexlib.Decoder(SHAPE, w, X, batch=1, max_ctx=96, max_new=T)
    try:
        dec.prefill(0, prompt)
        return dec.generate()[0]
    finally:
        if own:
            dec.close()


def test_bounded_wait_timeout_is_reported_and_handle_survives():
    dexlib = require_gpu()
    w = di.gen_weights(SHAPE, 0.3, seed=0, device="cuda")
    prompt = di.gen_prompts(SHAPE, 1, 20)[0].tolist()
    want = _decode(dexlib, w, prompt, 12)
    dec = dexlib.Decoder(SHAPE, w, X, batch=1, max_ctx=96, max_new=12)
    try:
        assert dec.selftest_stall(1000) == dexlib.DEX_ETIMEOUT
        # the flag was consumed by the check: a second stall is reported again, not stuck
        assert dec.selftest_stall(2000) == dexlib.DEX_ETIMEOUT
        assert dec.selftest_stall(0) == dexlib.DEX_EINVAL
        # the handle decodes as a fresh one does
        assert _decode(dexlib, w, prompt, 12, dec) == want
        # and a stall in the middle of a request does not disturb what follows
        dec.prefill(0, prompt)
        first, _ = dec.step()
        assert dec.selftest_stall(1000) == dexlib.DEX_ETIMEOUT
        assert _decode(dexlib, w, prompt, 12, dec) == want
    finally:
        dec.close()


def _free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


@pytest.mark.parametrize("fail_at", [1, 3, 12, 22])
def test_injected_allocation_failure_returns_enomem_without_leaks(fail_at):
    dexlib = require_gpu()
    w = di.gen_weights(SHAPE, 0.3, seed=0, device="cuda")
    cfg = dict(batch=2, max_ctx=96, max_new=8)
    # a successful handle first: loads every kernel module, so later free-memory readings
    # only move with the handle's own buffers
    dexlib.Decoder(SHAPE, w, X, **cfg).close()
    before = _free_bytes()
    os.environ["DEX_FAIL_ALLOC_AT"] = str(fail_at)
    try:
        with pytest.raises(dexlib.DexError) as e:
            dexlib.Decoder(SHAPE, w, X, **cfg)
        assert e.value.code == dexlib.DEX_ENOMEM
    finally:
        del os.environ["DEX_FAIL_ALLOC_AT"]
    assert _free_bytes() == before
    # without the injection the same call succeeds and decodes
    prompt = di.gen_prompts(SHAPE, 1, 20)[0].tolist()
    assert len(_decode(dexlib, w, prompt, 8)) == 8

"""GPU parity of the kernels in isolation against the fp64 oracle / closed forms.

* exit head + DECS (tcgen05 GEMM with the EXIT epilogue): logits vs RMSNorm(h) W^T in
  fp64, tokens vs Algorithm 2 on the oracle's logits wherever the decision margin > 0.1;
* KV collapse gather/scatter: bit-exact against the closed-form index map.
"""
import numpy as np
import pytest
import torch

import dex_inputs as di
from gpu_util import require_gpu
from oracle import dex as odex
from oracle.model import rmsnorm, widen_bf16

pytestmark = pytest.mark.gpu


def exit_case_inputs(n_slots, depth, d, V, seed=3, std=0.02):
    """Hidden rows, LM head, node table and DECS priors for an isolated exit-head call.

    Node k of a slot chain masks the oracle's top-k tokens of its slot, so the mask acts
    on the argmax itself; the last node of each chain is the unmasked reference.
    """
    m = di.ExitMicro(n_slots=n_slots, depth=depth, d_model=d, vocab=V, seed=seed, std=std)
    h, w = di.gen_exit_micro(m, device="cuda")
    hh = widen_bf16(di.bf16_bits(h))
    ww = widen_bf16(di.bf16_bits(w))
    z = rmsnorm(hh, np.ones(d), 1e-5) @ ww.T
    nodes, priors = [], []
    for s in range(n_slots):
        top = np.argsort(-z[s * depth])[:depth].tolist()
        for k in range(depth):
            unmasked = 1 if k == depth - 1 else 0
            pr = [] if unmasked else top[:k]
            nodes.append((s, 100 + s, unmasked, len(priors), len(pr)))
            priors += pr
    return h, w, z, nodes, priors


def check_exit_tokens(toks, z, nodes, priors, rule):
    checked = 0
    for i, (s, pos, unm, off, cnt) in enumerate(nodes):
        zz = z[i].copy()
        for v in priors[off:off + cnt]:
            zz[v] = -np.inf
        score = odex.decision_scores(zz, rule, s, pos)
        if odex.margin(score) > 0.1:
            assert toks[i] == odex.first_argmax(score), (i, toks[i], odex.first_argmax(score))
            checked += 1
        assert toks[i] not in priors[off:off + cnt]
    return checked


def _exit_case(n_slots, depth, d, V, sample, tau=0.7, std=0.02):
    dexlib = require_gpu()
    h, w, z, nodes, priors = exit_case_inputs(n_slots, depth, d, V, std=std)
    n = n_slots * depth
    g = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    nodes_t = torch.tensor(nodes, dtype=torch.int32, device="cuda")
    priors_t = torch.tensor(priors + [0], dtype=torch.int32, device="cuda")
    tokens = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    logits = torch.zeros((n, V), dtype=torch.float32, device="cuda")
    dexlib.dex_exit_head_decs(h.data_ptr(), n, d, g.data_ptr(), 1e-5, w.data_ptr(), V, nodes_t.data_ptr(),
                              priors_t.data_ptr(), sample, tau, 1234, tokens.data_ptr(), logits.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    gl = logits.cpu().numpy().astype(np.float64)
    err = float(np.max(np.abs(gl - z)))
    assert err < 2e-3 * max(1.0, float(np.abs(z).max()) / 8), f"exit logits max-abs error {err}"
    checked = check_exit_tokens(tokens.cpu().tolist(), z, nodes, priors, odex.Rule(sample=sample, tau=tau, seed=1234))
    assert checked >= n // 2
    return err


@pytest.mark.parametrize("sample", [False, True])
def test_exit_head_decs_small_ragged(sample):
    # vocab 1000 is not a multiple of the 128-row tile; d = 256 uses 4 k-blocks.  A wider
    # head (std 0.2) keeps the decision margins above 0.1 for most nodes at this small d.
    _exit_case(n_slots=3, depth=4, d=256, V=1000, sample=sample, std=0.2)


@pytest.mark.parametrize("sample", [False, True])
def test_exit_head_decs_split_k(sample):
    # few vocab tiles -> fixed split-K with the last-arriving CTA reducing partials
    _exit_case(n_slots=4, depth=5, d=2048, V=2048, sample=sample)


@pytest.mark.parametrize("sample", [False, True])
def test_exit_head_decs_microbench_size(sample):
    # kernel micro-benchmark shape: 64 nodes = 8 slot chains x 8 depths, LM head 128256 x 4096
    _exit_case(n_slots=8, depth=8, d=4096, V=128256, sample=sample)


def test_kv_collapse_bit_exact():
    dexlib = require_gpu()
    B, L, KVH, hd, ctx, S = 2, 32, 8, 128, 4096, 8
    gen = torch.Generator(device="cuda").manual_seed(0)
    committed = torch.randn((B, L, 2, KVH, ctx, hd), generator=gen, device="cuda").to(torch.bfloat16)
    pool = torch.randn((B, S, L, 2, KVH, hd), generator=gen, device="cuda").to(torch.bfloat16)
    jobs = [(0, 3, 4000, 32), (1, 5, 17, 12), (1, 0, 4095, 1), (0, 7, 0, 7), (1, 2, 2048, 32), (0, 1, 1, 20)]
    # out-of-range jobs (sequence, slot, position, layer count) are skipped and counted;
    # the kernel checks every field before any access
    bad = [(B, 0, 0, 1), (-1, 0, 0, 1), (0, S, 0, 1), (0, 0, ctx, 1), (0, 0, -3, 1), (0, 0, 5, L + 1),
           (0, 0, 5, 0)]
    before = committed.clone()
    jt = torch.tensor(jobs[:3] + bad + jobs[3:], dtype=torch.int32, device="cuda")
    rejected = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    geom = dexlib.dex_kv_geom(B, L, KVH, hd, ctx, S)
    dexlib.dex_kv_collapse(committed.data_ptr(), pool.data_ptr(), geom, jt.data_ptr(), jt.shape[0],
                           torch.cuda.current_stream().cuda_stream, rejected.data_ptr())
    torch.cuda.synchronize()
    want = before.clone()
    for seq, slot, pos, nl in jobs:
        want[seq, :nl, :, :, pos, :] = pool[seq, slot, :nl]
    assert torch.equal(committed.view(torch.int16), want.view(torch.int16))
    assert int(rejected.item()) == len(bad)
    # a bad geometry is refused on the host
    with pytest.raises(dexlib.DexError):
        dexlib.dex_kv_collapse(committed.data_ptr(), pool.data_ptr(), dexlib.dex_kv_geom(0, L, KVH, hd, ctx, S),
                               jt.data_ptr(), 1, torch.cuda.current_stream().cuda_stream)

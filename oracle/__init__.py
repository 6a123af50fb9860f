"""CPU oracle for Depth Exploration Decoding (DEX) -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 restatement of what the GPU library computes, written from
"Depth Exploration for LLM Decoding" (arXiv 2606.29223):

* ``analysis``  -- the depth-readiness quantities of section 2 (Eq. 1-14, Def. 1-5,
                   Prop. 3, 6, 7 and the worked examples of Appendix A.2/A.3);
* ``philox``    -- Philox4x32-10 (Salmon et al., SC'11) and the Gumbel(0,1) rows
                   that the sampling rule and DECS draw from;
* ``model``     -- the Llama-style pre-norm decoder (RMSNorm, RoPE, causal softmax
                   attention with GQA, SwiGLU FFN) and the shared exit head;
* ``dex``       -- autoregressive decoding, depth exploration decoding as the
                   section 3.2 prose describes it (exploration cycles, commit,
                   collapse), depth-coupled sampling (section 3.3) and the
                   brute-force EAD measurement.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  It shares no code with ``lossless_depth_adaptive_gb300`` and
never imports it; the two meet only through the seeded inputs of ``dex_inputs``.

Every function is pinned by a ``-m "not gpu"`` test against the paper's worked
examples, closed forms, invariants or an independent library routine; there is no
"parity unpinned" function in this package.
"""

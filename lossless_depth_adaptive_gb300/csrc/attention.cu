// Lattice-masked decode attention for a stage batch of DEX nodes.
//
// A node at input position p attends keys 0..p of its own token prefix (section 3.2:
// "ancestry, KV entries, and attention masks" follow the binary lattice).  Keys at
// positions < c_end come from the committed cache (shared by every node of the
// sequence); keys at c_end..p are the branch entries of the node's P-ancestors' slot
// chains and its own, read from the branch pool through the node's tail table.
//
// Work split: CTA = (sequence item, KV head, 128-position key group).  The committed
// keys and values of the group are staged once in shared memory by two bulk copies and
// reused by every node and every query head of the KV head (GQA).  Each warp owns a
// 32-key slice of the group for every query.  The arithmetic for a query is fixed by
// absolute positions only -- 32-key slices aligned to position 0, slices combined in
// order within the group, 128-position groups combined in group order by the last CTA
// to finish -- so a node's output is bit-identical whether its keys sit in the
// committed cache or the branch pool and whatever batch it is computed in.
#include "common.cuh"
#include "kernels.h"

namespace dex {

constexpr int kAttnThreads = 128;
constexpr int kGroupPos = 128;

// q . k for one fp32 key row.  The 16-byte chunks of the row are visited starting at
// chunk `rot` (the lane's index), so the lanes of a quarter-warp reading different key
// rows of an unpadded shared-memory tile hit distinct banks; four independent partial
// sums shorten the dependency chain.  The visiting order and the summation tree are
// functions of the key's absolute position only (lane = position mod 32), so a key's
// score does not depend on where the key is stored or which batch it is computed in.
template <int HD>
__device__ __forceinline__ float dot_q_row(const float* q, const float* krow, int rot) {
  constexpr int NC = HD / 4;
  float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = (i + rot) & (NC - 1);
    const float4 k4 = *reinterpret_cast<const float4*>(krow + c * 4);
    const float4 q4 = *reinterpret_cast<const float4*>(q + c * 4);
    float& a = s[i & 3];
    a = fmaf(q4.x, k4.x, a);
    a = fmaf(q4.y, k4.y, a);
    a = fmaf(q4.z, k4.z, a);
    a = fmaf(q4.w, k4.w, a);
  }
  return __fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3]));
}

constexpr int kQBatch = 8;    // queries staged per pass

template <int HD>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
  constexpr int DPL = HD / 32;        // output dims per lane
  constexpr int PS = HD + 2;          // partial record: acc[HD], m, l
  extern __shared__ __align__(128) uint8_t smem_raw[];
  float* sK = reinterpret_cast<float*>(smem_raw);   // [128][HD] fp32, unpadded
  float* sV = sK + kGroupPos * HD;
  float* sQ = reinterpret_cast<float*>(sV + kGroupPos * HD);         // [kQBatch][HD]
  float* sP = sQ + kQBatch * HD;                                     // [kQBatch][4 warps][PS]
  __shared__ int s_last;
  __shared__ __align__(8) uint64_t s_bar;

  const int g = blockIdx.x, kvh = blockIdx.y, it = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  const AttnItem item = a.items[it];
  if (g >= item.n_groups) return;
  const int g0 = g * kGroupPos;
  const int H = a.H, G = a.H / a.KVH;

  // committed keys/values of positions [g0, cmax) for this KV head: two contiguous
  // bulk copies (head-major cache: a head's positions are consecutive HD-element rows)
  const int cmax = min(g0 + kGroupPos, item.max_cend);
  if (cmax > g0) {
    if (tid == 0) {
      const size_t kbase =
          ((((static_cast<size_t>(item.seq) * a.L + item.layer) * 2 + 0) * a.KVH + kvh) * a.max_ctx + g0) * HD;
      const size_t vbase =
          ((((static_cast<size_t>(item.seq) * a.L + item.layer) * 2 + 1) * a.KVH + kvh) * a.max_ctx + g0) * HD;
      const uint32_t bytes = static_cast<uint32_t>(cmax - g0) * HD * 4;
      mbar_arrive_expect_tx(&s_bar, 2 * bytes);
      bulk_load_1d(sK, a.kv_commit + kbase, bytes, &s_bar);
      bulk_load_1d(sV, a.kv_commit + vbase, bytes, &s_bar);
    }
    if (!mbar_wait(&s_bar, 0, a.err, DEV_TIMEOUT_FULL)) {
      mbar_wait(&s_bar, 0, nullptr, 0);   // the copies may still land: wait (bounded) before exiting
      return;
    }
  }

  const int nq = (item.row_end - item.row_begin) * G;
  const int ks = g0 + 32 * warp;       // this warp's 32-key slice
  const int k = ks + lane;             // this lane's key
  for (int qb = 0; qb < nq; qb += kQBatch) {
    const int nb = min(kQBatch, nq - qb);
    for (int idx = tid; idx < nb * HD; idx += kAttnThreads) {
      const int qi = qb + idx / HD, d = idx % HD;
      const int row = item.row_begin + qi / G, qh = kvh * G + qi % G;
      sQ[idx] = a.q[(static_cast<size_t>(row) * H + qh) * HD + d] * a.scale_log2;
    }
    __syncthreads();
    // each warp: its 32-key slice against every query of the batch
    for (int j = 0; j < nb; ++j) {
      const int qi = qb + j;
      const DevNode nd = a.nodes[item.row_begin + qi / G];
      const int pos = nd.pos, c_end = nd.c_end;
      auto key_row = [&](int kk, int kv) -> const float* {
        if (kk < c_end) return (kv ? sV : sK) + (kk - g0) * HD;
        int t = kk - c_end;
        if (t >= nd.n_tail) {   // cannot happen for a well-formed plan; never read out of bounds
          atomicExch(a.err, DEV_BAD_INDEX);
          t = nd.n_tail - 1;
        }
        const int slot = a.tails[nd.tail_off + t];
        return a.kv_pool +
               ((((static_cast<size_t>(nd.seq) * a.n_slots + slot) * a.L + item.layer) * 2 + kv) * a.KVH + kvh) * HD;
      };
      const float s = (k <= pos) ? dot_q_row<HD>(sQ + j * HD, key_row(k, 0), lane) : -INFINITY;
      const float m = warp_max(s);
      float l = 0.0f, acc[DPL];
#pragma unroll
      for (int i = 0; i < DPL; ++i) acc[i] = 0.0f;
      if (m != -INFINITY) {
        const float p = exp2f(s - m);
        l = warp_sum(p);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          if (ks + jj <= pos) {   // uniform across the warp
            const float pk = __shfl_sync(0xffffffffu, p, jj);
            const float* vr = key_row(ks + jj, 1);
            if constexpr (DPL == 4) {
              const float4 f = *reinterpret_cast<const float4*>(vr + lane * 4);
              acc[0] = fmaf(pk, f.x, acc[0]);
              acc[1] = fmaf(pk, f.y, acc[1]);
              acc[2] = fmaf(pk, f.z, acc[2]);
              acc[3] = fmaf(pk, f.w, acc[3]);
            } else {
              const float2 f = *reinterpret_cast<const float2*>(vr + lane * 2);
              acc[0] = fmaf(pk, f.x, acc[0]);
              acc[1] = fmaf(pk, f.y, acc[1]);
            }
          }
        }
      }
      float* rec = sP + (j * 4 + warp) * PS;
#pragma unroll
      for (int i = 0; i < DPL; ++i) rec[lane * DPL + i] = acc[i];
      if (lane == 0) {
        rec[HD] = m;
        rec[HD + 1] = l;
      }
    }
    __syncthreads();
    // combine the four slices of each query in slice order; write the group's record
    for (int j = warp; j < nb; j += 4) {
      const int qi = qb + j;
      const int row = item.row_begin + qi / G, qh = kvh * G + qi % G;
      const float* r0 = sP + (j * 4) * PS;
      float mw[4], wgt[4];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        mw[w] = r0[w * PS + HD];
        M = fmaxf(M, mw[w]);
      }
#pragma unroll
      for (int w = 0; w < 4; ++w) wgt[w] = (mw[w] == -INFINITY) ? 0.0f : exp2f(mw[w] - M);
      const float Lg = __fadd_rn(__fadd_rn(r0[0 * PS + HD + 1] * wgt[0], r0[1 * PS + HD + 1] * wgt[1]),
                                 __fadd_rn(r0[2 * PS + HD + 1] * wgt[2], r0[3 * PS + HD + 1] * wgt[3]));
      float* pp = a.part + ((static_cast<size_t>(row) * H + qh) * a.max_groups + g) * PS;
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        const int d = lane * DPL + i;
        const float v = __fadd_rn(__fadd_rn(r0[0 * PS + d] * wgt[0], r0[1 * PS + d] * wgt[1]),
                                  __fadd_rn(r0[2 * PS + d] * wgt[2], r0[3 * PS + d] * wgt[3]));
        __stcg(pp + d, v);
      }
      if (lane == 0) {
        __stcg(pp + HD, M);
        __stcg(pp + HD + 1, Lg);
      }
    }
    __syncthreads();
  }

  // the last group CTA of (item, KV head) merges the groups; lane gg holds group gg
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.counters + item.counter * a.KVH + kvh, 1) == item.n_groups - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int qi = warp; qi < nq; qi += 4) {
    const int row = item.row_begin + qi / G, qh = kvh * G + qi % G;
    const float* base = a.part + (static_cast<size_t>(row) * H + qh) * a.max_groups * PS;
    float mg = -INFINITY, lg = 0.0f;
    if (lane < item.n_groups) {
      mg = __ldcg(base + lane * PS + HD);
      lg = __ldcg(base + lane * PS + HD + 1);
    }
    const float M = warp_max(mg);
    const float wg = (lg > 0.0f) ? exp2f(mg - M) : 0.0f;
    const float Lsum = warp_sum(lg * wg);
    float O[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) O[i] = 0.0f;
    for (int gg = 0; gg < item.n_groups; ++gg) {
      const float w = __shfl_sync(0xffffffffu, wg, gg);
      if (w == 0.0f) continue;
#pragma unroll
      for (int i = 0; i < DPL; ++i) O[i] = fmaf(w, __ldcg(base + gg * PS + lane * DPL + i), O[i]);
    }
    const float invl = 1.0f / Lsum;
    const size_t lo = static_cast<size_t>(a.plane_rows) * H * HD;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const size_t o = static_cast<size_t>(row) * H * HD + qh * HD + lane * DPL + i;
      store_pair(a.out + o, a.out + lo + o, O[i] * invl);
    }
  }
  if (tid == 0) a.counters[item.counter * a.KVH + kvh] = 0;
}

static size_t attn_smem_bytes(int hd) {
  return static_cast<size_t>(2) * kGroupPos * hd * 4 + kQBatch * hd * 4 + kQBatch * 4 * (hd + 2) * 4;
}

cudaError_t launch_attention(const AttnArgs& a, int n_items, int max_groups_launch, cudaStream_t st, bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  if (!a.nodes || !a.items || !a.tails || !a.q || !a.kv_commit || !a.kv_pool || !a.out || !a.part || !a.counters ||
      !a.err || a.plane_rows < 1 || max_groups_launch < 1 || max_groups_launch > a.max_groups || max_groups_launch > 32)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(max_groups_launch), static_cast<unsigned>(a.KVH),
                     static_cast<unsigned>(n_items));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.hd == 128) {
    cfg.dynamicSmemBytes = attn_smem_bytes(128);
    static bool set = false;
    if (!set) {
      cudaError_t e = cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(cfg.dynamicSmemBytes));
      if (e != cudaSuccess) return e;
      set = true;
    }
    return cudaLaunchKernelEx(&cfg, attn_kernel<128>, a);
  }
  if (a.hd == 64) {
    cfg.dynamicSmemBytes = attn_smem_bytes(64);
    static bool set = false;
    if (!set) {
      cudaError_t e = cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(cfg.dynamicSmemBytes));
      if (e != cudaSuccess) return e;
      set = true;
    }
    return cudaLaunchKernelEx(&cfg, attn_kernel<64>, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dex

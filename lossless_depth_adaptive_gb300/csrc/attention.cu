// Lattice-masked decode attention for a stage batch of DEX nodes.
//
// A node at input position p attends keys 0..p of its own token prefix (section 3.2:
// "ancestry, KV entries, and attention masks" follow the binary lattice).  Keys at
// positions < c_end come from the committed cache (shared by every node of the
// sequence); keys at c_end..p are the branch entries of the node's P-ancestors' slot
// chains and its own, read from the branch pool through the node's tail table.
//
// Work split: CTA = (sequence item, KV head, 128-position key group).  The committed
// keys of the group are staged once in shared memory and reused by every node and
// every query head of the KV head (GQA).  The arithmetic for a query is fixed by
// absolute positions only -- 64-key chunks aligned to position 0, a per-chunk
// softmax merged in chunk order, 128-position groups merged in group order by the
// last CTA to finish -- so a node's output is bit-identical whether its keys sit in
// the committed cache or the branch pool and whatever batch it is computed in.
#include "common.cuh"
#include "kernels.h"

namespace dex {

constexpr int kAttnThreads = 128;
constexpr int kGroupPos = 128;
constexpr int kChunkPos = 64;

template <int HD>
__device__ __forceinline__ float dot_q_row(const float* q, const __nv_bfloat16* krow) {
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < HD / 8; ++c) {
    const uint4 raw = *reinterpret_cast<const uint4*>(krow + c * 8);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h2[e]);
      s = fmaf(q[c * 8 + 2 * e], f.x, s);
      s = fmaf(q[c * 8 + 2 * e + 1], f.y, s);
    }
  }
  return s;
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
  constexpr int RS = HD + 8;          // padded smem row (bf16 elements)
  constexpr int DPL = HD / 32;        // output dims per lane
  extern __shared__ uint8_t smem_raw[];
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* sV = sK + kGroupPos * RS;
  float* sQ = reinterpret_cast<float*>(sV + kGroupPos * RS);   // [4 warps][HD]
  __shared__ int s_last;

  const int g = blockIdx.x, kvh = blockIdx.y, it = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_wait();
  griddep_launch_dependents();
  const AttnItem item = a.items[it];
  if (g >= item.n_groups) return;
  const int g0 = g * kGroupPos;
  const int H = a.H, G = a.H / a.KVH;

  // stage committed keys/values of positions [g0, cmax) for this KV head
  const int cmax = min(g0 + kGroupPos, item.max_cend);
  const size_t head_base_k =
      (((static_cast<size_t>(item.seq) * a.L + a.layer) * 2 + 0) * a.KVH + kvh) * a.max_ctx * HD;
  const size_t head_base_v =
      (((static_cast<size_t>(item.seq) * a.L + a.layer) * 2 + 1) * a.KVH + kvh) * a.max_ctx * HD;
  for (int idx = tid; idx < (cmax - g0) * (HD / 8); idx += kAttnThreads) {
    const int p = idx / (HD / 8), ch = idx % (HD / 8);
    const size_t off = static_cast<size_t>(g0 + p) * HD + ch * 8;
    *reinterpret_cast<uint4*>(sK + p * RS + ch * 8) = *reinterpret_cast<const uint4*>(a.kv_commit + head_base_k + off);
    *reinterpret_cast<uint4*>(sV + p * RS + ch * 8) = *reinterpret_cast<const uint4*>(a.kv_commit + head_base_v + off);
  }
  __syncthreads();

  const int nrows = item.row_end - item.row_begin;
  const int nq = nrows * G;
  float* q = sQ + warp * HD;
  for (int qi = warp; qi < nq; qi += 4) {
    const int row = item.row_begin + qi / G;
    const int qh = kvh * G + qi % G;
    const DevNode nd = a.nodes[row];
    const int pos = nd.pos, c_end = nd.c_end;
    for (int d = lane; d < HD; d += 32) q[d] = a.q[(static_cast<size_t>(row) * H + qh) * HD + d] * a.scale_log2;
    __syncwarp();
    auto branch_row = [&](int k, int kv) -> const __nv_bfloat16* {
      int t = k - c_end;
      if (t >= nd.n_tail) {   // cannot happen for a well-formed plan; never read out of bounds
        atomicExch(a.err, DEV_BAD_INDEX);
        t = nd.n_tail - 1;
      }
      const int slot = a.tails[nd.tail_off + t];
      return a.kv_pool +
             ((((static_cast<size_t>(nd.seq) * a.n_slots + slot) * a.L + a.layer) * 2 + kv) * a.KVH + kvh) * HD;
    };
    float m = -INFINITY, l = 0.0f, acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.0f;
    for (int c = g0; c < g0 + kGroupPos && c <= pos; c += kChunkPos) {
      float s[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int k = c + lane + 32 * t;
        if (k > pos) {
          s[t] = -INFINITY;
        } else {
          const __nv_bfloat16* kr = k < c_end ? sK + (k - g0) * RS : branch_row(k, 0);
          s[t] = dot_q_row<HD>(q, kr);
        }
      }
      const float mc = warp_max(fmaxf(s[0], s[1]));
      const float p0 = exp2f(s[0] - mc), p1 = exp2f(s[1] - mc);
      const float lc = warp_sum(p0 + p1);
      float accc[DPL];
#pragma unroll
      for (int i = 0; i < DPL; ++i) accc[i] = 0.0f;
      const int kend = min(c + kChunkPos - 1, pos);
      for (int k = c; k <= kend; ++k) {
        const float mine = (k - c) < 32 ? p0 : p1;
        const float pk = __shfl_sync(0xffffffffu, mine, (k - c) & 31);
        const __nv_bfloat16* vr = k < c_end ? sV + (k - g0) * RS : branch_row(k, 1);
        if (DPL == 4) {
          const uint2 raw = *reinterpret_cast<const uint2*>(vr + lane * 4);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
          const float2 f0 = __bfloat1622float2(h2[0]), f1 = __bfloat1622float2(h2[1]);
          accc[0] = fmaf(pk, f0.x, accc[0]);
          accc[1] = fmaf(pk, f0.y, accc[1]);
          accc[2] = fmaf(pk, f1.x, accc[2]);
          accc[3] = fmaf(pk, f1.y, accc[3]);
        } else {
          const __nv_bfloat162 h2 = *reinterpret_cast<const __nv_bfloat162*>(vr + lane * 2);
          const float2 f0 = __bfloat1622float2(h2);
          accc[0] = fmaf(pk, f0.x, accc[0]);
          accc[1] = fmaf(pk, f0.y, accc[1]);
        }
      }
      const float mn = fmaxf(m, mc);
      const float sa = exp2f(m - mn), sb = exp2f(mc - mn);
      l = l * sa + lc * sb;
#pragma unroll
      for (int i = 0; i < DPL; ++i) acc[i] = acc[i] * sa + accc[i] * sb;
      m = mn;
    }
    float* pp = a.part + ((static_cast<size_t>(row) * H + qh) * a.max_groups + g) * (HD + 2);
#pragma unroll
    for (int i = 0; i < DPL; ++i) __stcg(pp + lane * DPL + i, acc[i]);
    if (lane == 0) {
      __stcg(pp + HD, m);
      __stcg(pp + HD + 1, l);
    }
    __syncwarp();
  }

  // the last group CTA of (item, KV head) merges the groups in order
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.counters + item.counter * a.KVH + kvh, 1) == item.n_groups - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int qi = warp; qi < nq; qi += 4) {
    const int row = item.row_begin + qi / G;
    const int qh = kvh * G + qi % G;
    float M = -INFINITY, Lsum = 0.0f, O[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) O[i] = 0.0f;
    for (int gg = 0; gg < item.n_groups; ++gg) {
      const float* pp = a.part + ((static_cast<size_t>(row) * H + qh) * a.max_groups + gg) * (HD + 2);
      const float mg = __ldcg(pp + HD), lg = __ldcg(pp + HD + 1);
      if (lg == 0.0f) continue;   // no visible key in this group
      const float mn = fmaxf(M, mg);
      const float sa = exp2f(M - mn), sb = exp2f(mg - mn);
      Lsum = Lsum * sa + lg * sb;
#pragma unroll
      for (int i = 0; i < DPL; ++i) O[i] = O[i] * sa + __ldcg(pp + lane * DPL + i) * sb;
      M = mn;
    }
    const float invl = 1.0f / Lsum;
#pragma unroll
    for (int i = 0; i < DPL; ++i)
      a.out[static_cast<size_t>(row) * H * HD + qh * HD + lane * DPL + i] = __float2bfloat16_rn(O[i] * invl);
  }
  if (tid == 0) a.counters[item.counter * a.KVH + kvh] = 0;
}

cudaError_t launch_attention(const AttnArgs& a, int n_items, int max_groups_launch, cudaStream_t st, bool pdl) {
  if (n_items <= 0) return cudaSuccess;
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
    cfg.dynamicSmemBytes = 2 * kGroupPos * (128 + 8) * 2 + 4 * 128 * 4;
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
    cfg.dynamicSmemBytes = 2 * kGroupPos * (64 + 8) * 2 + 4 * 64 * 4;
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

// Lattice-masked decode attention for a stage batch of DEX nodes.
//
// A node at input position p attends keys 0..p of its own token prefix (section 3.2:
// "ancestry, KV entries, and attention masks" follow the binary lattice).  Keys at
// positions < c_end come from the committed cache (shared by every node of the
// sequence); keys at c_end..p are the branch entries of the node's P-ancestors' slot
// chains and its own, read from the branch pool through the node's tail table.
//
// Work split: CTA = (sequence item, KV head, 128-position key group); each warp owns a
// 32-key slice of the group, lane = key.  Keys and values are fp32 rows read straight
// from global memory (no shared-memory staging, so several CTAs share an SM and hide
// each other's latency): a lane walks its key's row in 16-byte chunks, and a key that is
// committed for every query of a batch is read once and scored against all of them.
// The arithmetic for a query is fixed by absolute positions only -- 32-key slices aligned
// to position 0, slices combined in order within the group, 128-position groups combined
// in group order by the last CTA to finish -- so a node's output is bit-identical whether
// its keys sit in the committed cache or the branch pool and whatever batch it is in.
#include "common.cuh"
#include "kernels.h"

namespace dex {

constexpr int kAttnThreads = 128;
constexpr int kGroupPos = 128;

// q . k for one fp32 key row.  The lane walks the row's 16-byte chunks starting at chunk
// `rot` (its index = key position mod 32) with four interleaved partial sums; the order is
// a function of the key's absolute position only.
template <int HD>
__device__ __forceinline__ float dot_q_row(const float* q, const float* krow, int rot) {
  constexpr int NC = HD / 4;
  float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int c = (i + rot) & (NC - 1);
    const float4 k4 = __ldg(reinterpret_cast<const float4*>(krow) + c);
    const float4 q4 = *reinterpret_cast<const float4*>(q + c * 4);
    float& a = s[i & 3];
    a = fmaf(q4.x, k4.x, a);
    a = fmaf(q4.y, k4.y, a);
    a = fmaf(q4.z, k4.z, a);
    a = fmaf(q4.w, k4.w, a);
  }
  return __fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3]));
}

constexpr int kQBatchMax = 8;  // largest query batch of a pass (QB is a template parameter: 1, 2, 4, 8)
constexpr int kVB = 8;         // value rows loaded ahead

// QB: queries per pass, chosen per launch from its largest item (the unused slots of a
// batch would otherwise still issue their predicated instructions).  A query's arithmetic
// is the same in every instantiation.
template <int HD, int QB>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
  constexpr int kQBatch = QB;
  constexpr int DPL = HD / 32;        // output dims per lane
  constexpr int NC = HD / 4;          // 16-byte chunks per row
  constexpr int PS = HD + 2;          // partial record: acc[HD], m, l
  extern __shared__ __align__(16) float smem_f[];
  float* sQ = smem_f;                 // [kQBatch][HD]
  float* sP = sQ + kQBatch * HD;      // [kQBatch][4 warps][PS]
  __shared__ int s_last;

  const int g = blockIdx.x, kvh = blockIdx.y, it = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_wait();
  griddep_launch_dependents();
  const AttnItem item = a.items[it];
  if (g >= item.n_groups) return;
  const int g0 = g * kGroupPos;
  const int H = a.H, G = a.H / a.KVH;
  // committed K and V rows of (sequence, layer, KV head): [max_ctx][HD] each
  const float* kcom =
      a.kv_commit + ((((static_cast<size_t>(item.seq) * a.L + item.layer) * 2 + 0) * a.KVH + kvh) * a.max_ctx) * HD;
  const float* vcom = kcom + static_cast<size_t>(a.KVH) * a.max_ctx * HD;

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
    int pos[kQBatch], cend[kQBatch], nrow[kQBatch];
    int cend_min = 0x7fffffff, pos_max = -1;
#pragma unroll
    for (int j = 0; j < kQBatch; ++j) {
      pos[j] = -1;
      cend[j] = 0;
      nrow[j] = item.row_begin;
      if (j < nb) {
        nrow[j] = item.row_begin + (qb + j) / G;
        const DevNode* nd = a.nodes + nrow[j];
        pos[j] = nd->pos;
        cend[j] = nd->c_end;
        cend_min = min(cend_min, cend[j]);
        pos_max = max(pos_max, pos[j]);
      }
    }
    __syncthreads();
    // key (or value) row kk of query j: committed cache below its c_end, else the branch
    // entry of its P-ancestry from the pool through the node's tail table
    auto key_row = [&](int j, int kk, int kv) -> const float* {
      if (kk < cend[j]) return (kv ? vcom : kcom) + static_cast<size_t>(kk) * HD;
      const DevNode* nd = a.nodes + nrow[j];
      int t = kk - cend[j];
      if (t >= nd->n_tail) {   // cannot happen for a well-formed plan; never read out of bounds
        atomicExch(a.err, DEV_BAD_INDEX);
        t = nd->n_tail - 1;
      }
      const int slot = a.tails[nd->tail_off + t];
      return a.kv_pool +
             ((((static_cast<size_t>(item.seq) * a.n_slots + slot) * a.L + item.layer) * 2 + kv) * a.KVH + kvh) * HD;
    };
    // scores of this lane's key against every query of the batch
    float sc[kQBatch];
    if (k < cend_min && k <= pos_max) {   // committed for every query: read the row once
      float part[kQBatch][4];
#pragma unroll
      for (int j = 0; j < kQBatch; ++j) part[j][0] = part[j][1] = part[j][2] = part[j][3] = 0.0f;
      const float4* kr = reinterpret_cast<const float4*>(kcom + static_cast<size_t>(k) * HD);
#pragma unroll 16
      for (int i = 0; i < NC; ++i) {
        const int c = (i + lane) & (NC - 1);
        const float4 k4 = __ldg(kr + c);
#pragma unroll
        for (int j = 0; j < kQBatch; ++j) {
          if (j < nb) {
            const float4 q4 = *reinterpret_cast<const float4*>(sQ + j * HD + c * 4);
            float& acc = part[j][i & 3];
            acc = fmaf(q4.x, k4.x, acc);
            acc = fmaf(q4.y, k4.y, acc);
            acc = fmaf(q4.z, k4.z, acc);
            acc = fmaf(q4.w, k4.w, acc);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kQBatch; ++j)
        sc[j] = (j < nb && k <= pos[j]) ? __fadd_rn(__fadd_rn(part[j][0], part[j][1]), __fadd_rn(part[j][2], part[j][3]))
                                        : -INFINITY;
    } else {
#pragma unroll
      for (int j = 0; j < kQBatch; ++j)
        sc[j] = (j < nb && k <= pos[j]) ? dot_q_row<HD>(sQ + j * HD, key_row(j, k, 0), lane) : -INFINITY;
    }
    // per query: slice softmax statistics and the value accumulation, keys in order
    float mx[kQBatch], lsum[kQBatch], pr[kQBatch], acc[kQBatch][DPL];
#pragma unroll
    for (int j = 0; j < kQBatch; ++j) {
      mx[j] = warp_max(sc[j]);
      pr[j] = 0.0f;
      lsum[j] = 0.0f;
      if (mx[j] != -INFINITY) {
        pr[j] = exp2f(sc[j] - mx[j]);
        lsum[j] = warp_sum(pr[j]);
      }
#pragma unroll
      for (int i = 0; i < DPL; ++i) acc[j][i] = 0.0f;
    }
    // value rows in batches of kVB keys: a batch's loads are all issued before any is used
    for (int jb = 0; jb < 32; jb += kVB) {
      if (ks + jb > pos_max) break;   // uniform across the warp
      float vv[kVB][DPL];
#pragma unroll
      for (int u = 0; u < kVB; ++u) {
        const int key = ks + jb + u;
        const bool shared = key <= pos_max && key < cend_min;
        if constexpr (DPL == 4) {
          const float4 f = shared ? __ldg(reinterpret_cast<const float4*>(vcom + static_cast<size_t>(key) * HD) + lane)
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          vv[u][0] = f.x; vv[u][1] = f.y; vv[u][2] = f.z; vv[u][3] = f.w;
        } else {
          const float2 f = shared ? __ldg(reinterpret_cast<const float2*>(vcom + static_cast<size_t>(key) * HD) + lane)
                                  : make_float2(0.0f, 0.0f);
          vv[u][0] = f.x; vv[u][1] = f.y;
        }
      }
#pragma unroll
      for (int u = 0; u < kVB; ++u) {
        const int key = ks + jb + u, jj = jb + u;
        if (key <= pos_max) {       // uniform across the warp
          if (key < cend_min) {     // committed for every query: the row loaded above
#pragma unroll
            for (int j = 0; j < kQBatch; ++j) {
              if (j < nb && key <= pos[j]) {
                const float pk = __shfl_sync(0xffffffffu, pr[j], jj);
#pragma unroll
                for (int i = 0; i < DPL; ++i) acc[j][i] = fmaf(pk, vv[u][i], acc[j][i]);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < kQBatch; ++j) {
              if (j < nb && key <= pos[j]) {
                const float pk = __shfl_sync(0xffffffffu, pr[j], jj);
                const float* vr = key_row(j, key, 1) + lane * DPL;
#pragma unroll
                for (int i = 0; i < DPL; ++i) acc[j][i] = fmaf(pk, __ldg(vr + i), acc[j][i]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kQBatch; ++j) {
      if (j < nb) {
        float* rec = sP + (j * 4 + warp) * PS;
#pragma unroll
        for (int i = 0; i < DPL; ++i) rec[lane * DPL + i] = acc[j][i];
        if (lane == 0) {
          rec[HD] = mx[j];
          rec[HD + 1] = lsum[j];
        }
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

static size_t attn_smem_bytes(int hd, int qb) { return static_cast<size_t>(qb) * hd * 4 + qb * 4 * (hd + 2) * 4; }

template <int HD, int QB>
static cudaError_t launch_attn_variant(cudaLaunchConfig_t cfg, const AttnArgs& a) {
  static bool set = false;
  cfg.dynamicSmemBytes = attn_smem_bytes(HD, QB);
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<HD, QB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cfg.dynamicSmemBytes));
    if (e != cudaSuccess) return e;
    set = true;
  }
  return cudaLaunchKernelEx(&cfg, attn_kernel<HD, QB>, a);
}

template <int HD>
static cudaError_t launch_attn_hd(const cudaLaunchConfig_t& cfg, const AttnArgs& a, int max_nq) {
  if (max_nq <= 1) return launch_attn_variant<HD, 1>(cfg, a);
  if (max_nq <= 2) return launch_attn_variant<HD, 2>(cfg, a);
  if (max_nq <= 4) return launch_attn_variant<HD, 4>(cfg, a);
  return launch_attn_variant<HD, 8>(cfg, a);
}

cudaError_t launch_attention(const AttnArgs& a, int n_items, int max_groups_launch, int max_nq, cudaStream_t st,
                             bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  if (!a.nodes || !a.items || !a.tails || !a.q || !a.kv_commit || !a.kv_pool || !a.out || !a.part || !a.counters ||
      !a.err || a.plane_rows < 1 || max_groups_launch < 1 || max_groups_launch > a.max_groups ||
      max_groups_launch > 32 || max_nq < 1)
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
  if (a.hd == 128) return launch_attn_hd<128>(cfg, a, max_nq);
  if (a.hd == 64) return launch_attn_hd<64>(cfg, a, max_nq);
  return cudaErrorInvalidValue;
}

}  // namespace dex

// Lattice-masked decode attention for a stage batch of DEX nodes.
//
// A node at input position p attends keys 0..p of its own token prefix (section 3.2:
// "ancestry, KV entries, and attention masks" follow the binary lattice).  Keys at
// positions < c_end come from the committed cache (shared by every node of the
// sequence); keys at c_end..p are the branch entries of the node's P-ancestors' slot
// chains and its own, read from the branch pool through the node's tail table.
//
// Work split: CTA = (sequence item, KV head, 128-position key group), four warps, each
// owning a 32-key slice of the group.  Scores take lane = key: the group's committed key
// rows go to shared memory with asynchronous 16-byte copies (nothing held in registers,
// nothing through L1), chunk c of row r stored at chunk c ^ (r mod 32), so when every lane
// reads chunk c of its own row the 32 reads hit distinct banks while the query's chunk c
// is one broadcast read.  Values take lane = a run of output dimensions, so a warp reads
// one whole value row per load.  When the CTA's queries fit one pass (decode), the
// committed value rows follow the keys into the same shared buffer with a bulk copy once
// the scores are taken; otherwise (prefill) the key rows stay in shared memory across
// query batches and values are read from global memory eight rows ahead.  Branch keys
// (few per node) are read from the pool.  A committed key is read once and used for every
// query of the batch.
//
// The arithmetic for a query is fixed by absolute positions only -- 32-key slices aligned
// to position 0, each score summed in chunk order wherever the key row lives,
// slices combined in order within a group, groups combined in group order by the last
// CTA to finish -- so a node's output is bit-identical whether its keys sit in the
// committed cache or the branch pool and whatever batch it is in.
#include "common.cuh"
#include "kernels.h"

namespace dex {

constexpr int kAttnWarps = kAttnGroupPos / 32;
constexpr int kAttnThreads = 32 * kAttnWarps;
static_assert(kAttnGroupPos == 32 * kAttnWarps && kAttnWarps == 4, "four 32-key warp slices per group");
constexpr int kVB = 8;   // value rows loaded ahead

// q . k as four partial sums, one per feature residue mod 4 (features 4c + r go to sum r),
// accumulated over the chunks in order, two sums per packed FMA (each element rounded as
// fmaf), then (s0 + s1) + (s2 + s3).  The committed-key loop below follows the same order.
__device__ __forceinline__ void dot_chunk(float2& s01, float2& s23, const float4& q4, const float4& k4) {
  s01 = __ffma2_rn(make_float2(q4.x, q4.y), make_float2(k4.x, k4.y), s01);
  s23 = __ffma2_rn(make_float2(q4.z, q4.w), make_float2(k4.z, k4.w), s23);
}
__device__ __forceinline__ float dot_finish(const float2& s01, const float2& s23) {
  return __fadd_rn(__fadd_rn(s01.x, s01.y), __fadd_rn(s23.x, s23.y));
}

// Chunk c of the row sits at c ^ swz (shared-memory key rows are swizzled by row, pool rows
// are not).
template <int HD>
__device__ __forceinline__ float dot_q_row(const float* q, const float* krow, int swz) {
  constexpr int NC = HD / 4;
  float2 s01 = make_float2(0.0f, 0.0f), s23 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int c = 0; c < NC; ++c)
    dot_chunk(s01, s23, *reinterpret_cast<const float4*>(q + c * 4), *(reinterpret_cast<const float4*>(krow) + (c ^ swz)));
  return dot_finish(s01, s23);
}

// acc[i] += p * v[i] over the lane's output dims, two dims per packed FMA (each element
// rounded as fmaf, so the order per element is that of a scalar loop).
template <int DPL>
__device__ __forceinline__ void axpy_dims(float (&acc)[DPL], float p, const float (&v)[DPL]) {
  const float2 pp = make_float2(p, p);
#pragma unroll
  for (int i = 0; i < DPL; i += 2) {
    const float2 r = __ffma2_rn(pp, make_float2(v[i], v[i + 1]), make_float2(acc[i], acc[i + 1]));
    acc[i] = r.x;
    acc[i + 1] = r.y;
  }
}

// Shared floats of a CTA: key/value rows, queries and (unless SP) the slice records.
__host__ __device__ constexpr size_t attn_smem_floats(int hd, int qb, bool sp) {
  return static_cast<size_t>(kAttnGroupPos) * hd + static_cast<size_t>(qb) * hd +
         (sp ? 0 : static_cast<size_t>(qb) * kAttnWarps * (hd + 2));
}
static_assert(kAttnGroupPos * 64 >= 8 * kAttnWarps * (64 + 2), "slice records fit the key buffer");

// QB: queries per pass, chosen per launch from its largest item (the unused slots of a
// batch would otherwise still issue their predicated instructions).  SP: every item of the
// launch fits one pass, so the slice records reuse the key/value buffer once the values
// are consumed (a smaller CTA: three per SM instead of two).  A query's arithmetic is the
// same in every instantiation.
template <int HD, int QB, bool SP>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
  constexpr int DPL = HD / 32;        // output dims per lane
  constexpr int NC = HD / 4;          // 16-byte chunks per row
  constexpr int PS = HD + 2;          // partial record: acc[HD], m, l
  extern __shared__ __align__(128) float smem_f[];
  float* sK = smem_f;                             // [kAttnGroupPos][HD] committed keys of the group
  float* sQ = sK + kAttnGroupPos * HD;            // [QB][HD]
  float* sP = SP ? sK : sQ + QB * HD;             // [QB][warps][PS]
  __shared__ __align__(8) uint64_t vbar;          // value rows landed (single-pass CTAs)
  __shared__ int s_last;

  const int g = blockIdx.x, kvh = blockIdx.y, it = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_wait();   // q and this round's K/V come from the preceding launch
  griddep_launch_dependents();
  const AttnItem item = a.items[it];
  // the groups must cover every position up to max_pos (a malformed plan is reported)
  if (g == 0 && kvh == 0 && tid == 0 && item.n_groups * kAttnGroupPos <= item.max_pos) atomicExch(a.err, DEV_BAD_INDEX);
  if (g >= item.n_groups) return;
  const int g0 = g * kAttnGroupPos;
  const int H = a.H, G = a.H / a.KVH;
  // committed K and V rows of (sequence, layer, KV head): [max_ctx][HD] each
  const float* kcom =
      a.kv_commit + ((((static_cast<size_t>(item.seq) * a.L + item.layer) * 2 + 0) * a.KVH + kvh) * a.max_ctx) * HD;
  const float* vcom = kcom + static_cast<size_t>(a.KVH) * a.max_ctx * HD;
  // committed rows some query of the item reads: [g0, g0 + n_com)
  const int n_com = max(0, min(kAttnGroupPos, min(item.max_cend, item.max_pos + 1) - g0));
  if (tid == 0) {
    mbar_init(&vbar, 1);
    fence_mbar_init();
  }
  // committed key rows -> shared memory, chunk c of row r at c ^ (r mod NC): lanes reading
  // the same chunk of 32 consecutive rows hit distinct banks
  {
    const uint32_t base = smem_u32(sK);
    const float* src = kcom + static_cast<size_t>(g0) * HD;
    for (int idx = tid; idx < n_com * NC; idx += kAttnThreads) {
      const int r = idx / NC, c = idx % NC;
      cp_async_16(base + static_cast<uint32_t>(r * HD + ((c ^ (r & (NC - 1))) << 2)) * 4u, src + r * HD + c * 4);
    }
    cp_async_commit();
  }
  bool have_k = false, failed = false;

  const int nq = (item.row_end - item.row_begin) * G;
  if (SP && nq > QB) {   // the launch promised one pass per item
    if (tid == 0) atomicExch(a.err, DEV_BAD_INDEX);
    return;
  }
  // one query pass (decode): once scored, the key buffer takes the group's committed value
  // rows in one more bulk copy; several passes (prefill) keep the keys and read values from
  // global memory
  const bool v_smem = nq <= QB && n_com > 0;
  const int ks = g0 + 32 * warp;       // this warp's 32-key slice
  const int k = ks + lane;             // this lane's key
  for (int qb = 0; qb < nq; qb += QB) {
    const int nb = min(QB, nq - qb);
    for (int idx = tid; idx < nb * HD; idx += kAttnThreads) {
      const int qi = qb + idx / HD, d = idx % HD;
      const int row = item.row_begin + qi / G, qh = kvh * G + qi % G;
      sQ[idx] = a.q[(static_cast<size_t>(row) * H + qh) * HD + d] * a.scale_log2;
    }
    int pos[QB], cend[QB], nrow[QB];
    int cend_min = 0x7fffffff, pos_max = -1;
#pragma unroll
    for (int j = 0; j < QB; ++j) {
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
    __syncthreads();   // sQ written; the barriers' initialisation is visible
    if (!have_k) {
      cp_async_wait_all();
      __syncthreads();   // every thread's key chunks have landed
      have_k = true;
    }
    // the branch-pool row of query j's key kk (kk >= c_end of that query)
    auto pool_row = [&](int j, int kk, int kv) -> const float* {
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
    float sc[QB];
    if (k < cend_min && k <= pos_max) {   // committed for every query: one pass over the row
      float2 s01[QB], s23[QB];
#pragma unroll
      for (int j = 0; j < QB; ++j) s01[j] = s23[j] = make_float2(0.0f, 0.0f);
      const float4* kr = reinterpret_cast<const float4*>(sK + (k - g0) * HD);
      const int swz = (k - g0) & (NC - 1);
#pragma unroll 8
      for (int c = 0; c < NC; ++c) {
        const float4 k4 = kr[c ^ swz];
#pragma unroll
        for (int j = 0; j < QB; ++j) {
          // same address in every lane: broadcast
          if (j < nb) dot_chunk(s01[j], s23[j], *reinterpret_cast<const float4*>(sQ + j * HD + c * 4), k4);
        }
      }
#pragma unroll
      for (int j = 0; j < QB; ++j) sc[j] = (j < nb && k <= pos[j]) ? dot_finish(s01[j], s23[j]) : -INFINITY;
    } else {
#pragma unroll
      for (int j = 0; j < QB; ++j) {
        sc[j] = -INFINITY;
        if (j < nb && k <= pos[j])
          sc[j] = k < cend[j] ? dot_q_row<HD>(sQ + j * HD, sK + (k - g0) * HD, (k - g0) & (NC - 1))
                              : dot_q_row<HD>(sQ + j * HD, pool_row(j, k, 0), 0);
      }
    }
    if (v_smem) {
      __syncthreads();   // every score read of the key rows is done
      if (tid == 0) {
        const uint32_t bytes = static_cast<uint32_t>(n_com) * HD * 4;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&vbar, bytes);
        bulk_load_1d(sK, vcom + static_cast<size_t>(g0) * HD, bytes, &vbar);
      }
    }
    // per query: slice softmax statistics and the value accumulation, keys in order
    float mx[QB], lsum[QB], pr[QB], acc[QB][DPL];
#pragma unroll
    for (int j = 0; j < QB; ++j) {
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
    if (v_smem) {
      failed |= !mbar_wait(&vbar, 0, a.err, DEV_TIMEOUT_FULL);
      if (__syncthreads_or(failed)) {
        failed = true;
        break;
      }
      const int n_keys = min(32, pos_max - ks + 1);   // keys of the slice any query attends
#pragma unroll 4
      for (int u = 0; u < n_keys; ++u) {
        const int key = ks + u;
        const float* vs = sK + (key - g0) * HD + lane * DPL;
        if (key < cend_min) {   // committed for every query
          float vv[DPL];
          if constexpr (DPL == 4) {
            const float4 f = *reinterpret_cast<const float4*>(vs);
            vv[0] = f.x; vv[1] = f.y; vv[2] = f.z; vv[3] = f.w;
          } else {
            const float2 f = *reinterpret_cast<const float2*>(vs);
            vv[0] = f.x; vv[1] = f.y;
          }
#pragma unroll
          for (int j = 0; j < QB; ++j) {
            if (j < nb && key <= pos[j]) {
              const float pk = __shfl_sync(0xffffffffu, pr[j], u);
              axpy_dims<DPL>(acc[j], pk, vv);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < QB; ++j) {
            if (j < nb && key <= pos[j]) {
              const float pk = __shfl_sync(0xffffffffu, pr[j], u);
              const float* vr = key < cend[j] ? vs : pool_row(j, key, 1) + lane * DPL;
              float vt[DPL];
#pragma unroll
              for (int i = 0; i < DPL; ++i) vt[i] = vr[i];
              axpy_dims<DPL>(acc[j], pk, vt);
            }
          }
        }
      }
    } else {
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
            for (int j = 0; j < QB; ++j) {
              if (j < nb && key <= pos[j]) {
                const float pk = __shfl_sync(0xffffffffu, pr[j], jj);
                axpy_dims<DPL>(acc[j], pk, vv[u]);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < QB; ++j) {
              if (j < nb && key <= pos[j]) {
                const float pk = __shfl_sync(0xffffffffu, pr[j], jj);
                const float* vr =
                    (key < cend[j] ? vcom + static_cast<size_t>(key) * HD : pool_row(j, key, 1)) + lane * DPL;
                float vt[DPL];
#pragma unroll
                for (int i = 0; i < DPL; ++i) vt[i] = __ldg(vr + i);
                axpy_dims<DPL>(acc[j], pk, vt);
              }
            }
          }
        }
      }
    }
    }
    if constexpr (SP) __syncthreads();   // every warp is done with the value rows under sP
#pragma unroll
    for (int j = 0; j < QB; ++j) {
      if (j < nb) {
        float* rec = sP + (j * kAttnWarps + warp) * PS;
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
    for (int j = warp; j < nb; j += kAttnWarps) {
      const int qi = qb + j;
      const int row = item.row_begin + qi / G, qh = kvh * G + qi % G;
      const float* r0 = sP + (j * kAttnWarps) * PS;
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
  if (failed) return;   // error flag set; the host reports the stall

  // the last group CTA of (item, KV head) merges the groups; lane gg holds groups gg, gg + 32
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.counters + item.counter * a.KVH + kvh, 1) == item.n_groups - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int qi = warp; qi < nq; qi += kAttnWarps) {
    const int row = item.row_begin + qi / G, qh = kvh * G + qi % G;
    const float* base = a.part + (static_cast<size_t>(row) * H + qh) * a.max_groups * PS;
    float mg[2] = {-INFINITY, -INFINITY}, lg[2] = {0.0f, 0.0f};
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int gg = lane + 32 * h2;
      if (gg < item.n_groups) {
        mg[h2] = __ldcg(base + gg * PS + HD);
        lg[h2] = __ldcg(base + gg * PS + HD + 1);
      }
    }
    const float M = warp_max(fmaxf(mg[0], mg[1]));
    float wg[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) wg[h2] = (lg[h2] > 0.0f) ? exp2f(mg[h2] - M) : 0.0f;
    const float Lsum = warp_sum(__fadd_rn(lg[0] * wg[0], lg[1] * wg[1]));
    float O[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) O[i] = 0.0f;
    for (int gg = 0; gg < item.n_groups; ++gg) {
      const float w = __shfl_sync(0xffffffffu, gg < 32 ? wg[0] : wg[1], gg & 31);
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

template <int HD, int QB, bool SP>
static cudaError_t launch_attn_variant(cudaLaunchConfig_t cfg, const AttnArgs& a) {
  static bool set = false;
  cfg.dynamicSmemBytes = attn_smem_floats(HD, QB, SP) * 4;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<HD, QB, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cfg.dynamicSmemBytes));
    // three single-pass CTAs (about 69 KB each) fit only the largest shared-memory
    // configuration, which the driver does not choose by itself for these sizes
    if (e == cudaSuccess)
      e = (SP && smem_carveout_pref() < 0)
              ? cudaFuncSetAttribute(attn_kernel<HD, QB, SP>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     static_cast<int>(cudaSharedmemCarveoutMaxShared))
              : apply_carveout(attn_kernel<HD, QB, SP>);
    if (e != cudaSuccess) return e;
    set = true;
  }
  return cudaLaunchKernelEx(&cfg, attn_kernel<HD, QB, SP>, a);
}

template <int HD>
static cudaError_t launch_attn_hd(const cudaLaunchConfig_t& cfg, const AttnArgs& a, int max_nq) {
  if (max_nq <= 1) return launch_attn_variant<HD, 1, true>(cfg, a);
  if (max_nq <= 2) return launch_attn_variant<HD, 2, true>(cfg, a);
  if (max_nq <= 4) return launch_attn_variant<HD, 4, true>(cfg, a);
  if (max_nq <= 8) return launch_attn_variant<HD, 8, true>(cfg, a);
  return launch_attn_variant<HD, 8, false>(cfg, a);
}

cudaError_t launch_attention(const AttnArgs& a, int n_items, int max_groups_launch, int max_nq, cudaStream_t st,
                             bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  if (!a.nodes || !a.items || !a.tails || !a.q || !a.kv_commit || !a.kv_pool || !a.out || !a.part || !a.counters ||
      !a.err || a.plane_rows < 1 || max_groups_launch < 1 || max_groups_launch > a.max_groups ||
      max_groups_launch > kAttnMaxGroups || max_nq < 1 || (reinterpret_cast<uintptr_t>(a.kv_commit) & 15))
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

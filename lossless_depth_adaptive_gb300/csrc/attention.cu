// Lattice-masked attention for the node batches of a DEX round (and prefill chunks), with
// the bulk of every query's keys on the 5th-generation tensor cores.
//
// A node at input position p attends keys 0..p of its own token prefix (section 3.2:
// "ancestry, KV entries, and attention masks" follow the binary lattice).  Keys at
// positions < c_end come from the committed cache (shared by every node of the
// sequence); keys at c_end..p are the branch entries of the node's P-ancestors' slot
// chains and its own, read from the branch pool through the node's tail table.
//
// Split of a query's keys (fixed by its position p alone):
//  * bulk keys [0, b), b = max(0, p - kAttnWindow + 1): always committed (a node's branch
//    keys are its last <= |X| positions and kAttnWindow > |X|).  Per 128-position group,
//    scores S = K Q^T and the group output O = V^T P^T run as tcgen05 MMAs (M = 128 keys or
//    128 value dims, N = 16 queries) from shared-memory tiles: K and V fp16 tiles exactly as
//    cached, Q and P as fp16 hi/lo pairs (x ~= hi + lo, two MMAs into one fp32 accumulator),
//    so every product is carried to about fp32 precision.  A masked key gets p = 0, which
//    adds exact zeros.
//  * window keys [b, p] (at most kAttnWindow): fp32 dot products on CUDA cores, reading
//    the committed cache or the branch pool, in one fixed order wherever the row lives.
// The group partials (max, sum, output) are combined in group order and then with the
// window part by the unit that completes an (item, KV head).  A tensor-core element's
// value depends only on its own row and column operands, so a query's result is the same
// bits whatever else shares its MMA, whichever buffer holds its window keys, and whatever
// batch or launch it is in: GPU-DEX equals GPU-AR bit for bit.
//
// Work: a unit is (item, KV head, group); an item is one sequence's contiguous node rows of
// one layer (at most 16 queries per pass; prefill items take several passes).  Persistent
// CTAs (one per SM) take contiguous ranges of units.  Warp 0 streams the committed K and V
// tiles of each unit through a ring of shared-memory stages with TMA (128-byte swizzle,
// 32-row boxes); warp 1 owns TMEM and issues the MMAs; warps 2-5 build the query tiles,
// run the softmax between the two MMAs and write the group partials; the last two warps
// take the window keys and the final combinations of the (item, KV head)s off the critical
// path.
#include <cuda_fp16.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace dex {

constexpr int kQT = kAttnPassQueries;                 // queries per pass (MMA N)
constexpr int kMergeWarps = 2;
constexpr int kAttnThreads = 32 * (6 + kMergeWarps);  // producer, MMA, four epilogue warps, merge warps
constexpr int kBoxRows = 32;                          // TMA box height
constexpr int kEpiBar = 1, kMergeBar = 2;             // named barriers of the epilogue / merge warps
static_assert(kAttnGroupPos == 128 && kQT == 16, "128-key groups, 16-query MMA columns");

// Shared-memory plan: K/V ring; the query tile (rows 0-15 hi, 16-31 lo) and the
// probability tile (same); a zero atom that pads the 64-dim value tiles of head_dim 64 to
// the MMA's 128 rows; reduction scratch; barriers.
template <int HD>
struct AttnSmem {
  static constexpr uint32_t kTile = kAttnGroupPos * HD * 2;   // [128 rows][HD] fp16, HD/64 halves of 16 KB
  static constexpr uint32_t kStage = 2 * kTile;
  static constexpr int kStages = (HD == 128) ? 3 : 5;
  static constexpr uint32_t kRing = kStages * kStage;
  static constexpr uint32_t kQTile = 2 * kQT * HD * 2;          // [32][HD] fp16, HD/64 halves of 4 KB
  static constexpr uint32_t kPTile = 2 * kQT * kAttnGroupPos * 2;   // [32][128 keys] fp16, two halves of 4 KB
  static constexpr uint32_t kZero = (HD == 128) ? 0 : kAttnGroupPos * 128;
  static constexpr uint32_t oQ = kRing, oP = oQ + kQTile;
  static constexpr uint32_t oZero = oP + kPTile;
  static constexpr uint32_t oRed = oZero + kZero;                  // float [2][16][4] max / sum
  static constexpr uint32_t oMeta = oRed + 2 * 4 * kQT * 4;        // int [2][16] bulk bounds, int [2][16] record rows
  static constexpr uint32_t oBar = oMeta + 4 * kQT * 4 + 16;
  static constexpr uint32_t kTotal = oBar + (2 * kStages + 4) * 8 + 32 + 1024;   // + alignment slack
};

// MN-major operand descriptor, 128-byte swizzle: 64 contiguous 16-bit elements of M (or N)
// per 128-byte row, rows along K 128 bytes apart in 1024-byte 8-row atoms; lbo = bytes
// between 64-element atoms along M, sbo = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}
// kind::f16 instruction descriptor with fp16 A and B, fp32 D; a_mn: A is MN-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn) {
  return (1u << 4) | (a_mn ? (1u << 15) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// fp32 -> (hi, lo) fp16 pair: hi = fp16(x), lo = fp16(x - hi).
__device__ __forceinline__ void split_f16(float x, __half& hi, __half& lo) {
  hi = __float2half_rn(x);
  lo = __float2half_rn(__fsub_rn(x, __half2float(hi)));
}

// Byte offset of element (row, col) in a 128-byte-swizzled fp16 tile whose 64-column halves
// hold `rows` rows each.
__device__ __forceinline__ uint32_t sw_elem_off(int row, int col, int rows) {
  return static_cast<uint32_t>((col >> 6) * rows * 128 + row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) +
                               ((col & 7) << 1));
}

struct UnitRef {
  int item, kvh, g;
};
// Unit u of the launch: items are laid out back to back, KVH x n_groups units each.
__device__ __forceinline__ UnitRef unit_ref(const AttnArgs& a, int u) {
  int lo = 0, hi = a.n_items - 1;
  while (lo < hi) {   // last item with unit0 <= u
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&a.items[mid].unit0) <= u) lo = mid;
    else hi = mid - 1;
  }
  UnitRef r;
  r.item = lo;
  const int rem = u - __ldg(&a.items[lo].unit0);
  const int ng = __ldg(&a.items[lo].n_groups);
  r.kvh = rem / ng;
  r.g = rem - r.kvh * ng;
  return r;
}
__device__ __forceinline__ int bulk_end(int pos) { return max(0, pos - kAttnWindow + 1); }

// Walks a CTA's contiguous units in order without searching: the item record is reloaded
// only when the walk enters the next item.
struct UnitCursor {
  int item, kvh, g;
  AttnItem it;
  __device__ __forceinline__ void init(const AttnArgs& a, int u) {
    const UnitRef r = unit_ref(a, u);
    item = r.item;
    kvh = r.kvh;
    g = r.g;
    it = a.items[item];
  }
  __device__ __forceinline__ void next(const AttnArgs& a) {
    if (++g < it.n_groups) return;
    g = 0;
    if (++kvh < a.KVH) return;
    kvh = 0;
    if (++item < a.n_items) it = a.items[item];
  }
  __device__ __forceinline__ int n_queries(int G) const { return (it.row_end - it.row_begin) * G; }
};
// A cursor over the CTA's query passes (unit, pass within the unit).
struct PassCursor {
  UnitCursor c;
  int i, p;   // unit index within the CTA, pass within the unit
  __device__ __forceinline__ void init(const AttnArgs& a, int u0) {
    c.init(a, u0);
    i = 0;
    p = 0;
  }
  __device__ __forceinline__ void next(const AttnArgs& a, int G, int n_my) {
    if ((p + 1) * kQT < c.n_queries(G)) {
      ++p;
      return;
    }
    p = 0;
    if (++i < n_my) c.next(a);
  }
};

// Transposed butterfly over a warp for K (4, 8 or 16) values per lane: on return, the 32/K
// lanes 32j/K .. 32(j+1)/K - 1 hold the reduction over all 32 lanes of v[j] (K shuffles
// plus five minus log2 K, instead of K separate 5-step butterflies).  Whatever K, every
// lane's value is combined in the same tree -- pairs across lane bit 4, then bit 3, ...,
// then bit 0 -- so a query's sum is the same bits in a pass of 4, 8 or 16 columns.
template <int K, bool kMax>
__device__ __forceinline__ float warp_reduce_transposed(const float (&v)[K], int lane) {
  static_assert(K == 4 || K == 8 || K == 16, "4, 8 or 16 values per lane");
  auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : __fadd_rn(x, y); };
  float cur[K];
#pragma unroll
  for (int k = 0; k < K; ++k) cur[k] = v[k];
  int bit = 16;
#pragma unroll
  for (int w = K; w > 1; w >>= 1, bit >>= 1) {   // halve the values across lane bit `bit`
    const bool hi = lane & bit;
#pragma unroll
    for (int k = 0; k < w / 2; ++k) {
      const float send = hi ? cur[k] : cur[k + w / 2];
      const float keep = hi ? cur[k + w / 2] : cur[k];
      cur[k] = op(keep, __shfl_xor_sync(0xffffffffu, send, bit));
    }
  }
#pragma unroll
  for (; bit >= 1; bit >>= 1) cur[0] = op(cur[0], __shfl_xor_sync(0xffffffffu, cur[0], bit));
  return cur[0];
}

// Sum of the four accumulator chains of a product, hi and lo columns: for each query column
// j, v[j] = sum over chains c in order of (D_c[j] + D_c[j + 16]).
__device__ __forceinline__ void tmem_chain_sum(uint32_t taddr, float (&v)[kQT]) {
  uint32_t r0[32], r1[32];
#pragma unroll
  for (int c = 0; c < 4; c += 2) {
    tmem_ld32_nowait(taddr + static_cast<uint32_t>(c * 2 * kQT), r0);
    tmem_ld32_nowait(taddr + static_cast<uint32_t>((c + 1) * 2 * kQT), r1);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < kQT; ++j) {
      const float t0 = __fadd_rn(__uint_as_float(r0[j]), __uint_as_float(r0[j + kQT]));
      const float t1 = __fadd_rn(__uint_as_float(r1[j]), __uint_as_float(r1[j + kQT]));
      v[j] = (c == 0) ? __fadd_rn(t0, t1) : __fadd_rn(v[j], __fadd_rn(t0, t1));
    }
  }
}

// Window part of one query of an (item, KV head): keys [b, p] on CUDA cores, from the
// committed cache or the branch pool, stored as the query's record in the window slot of
// the partials (O unnormalised, max, sum).  One warp per query; the query's loads are issued
// before the arithmetic that needs them.
template <int HD>
__device__ __forceinline__ void window_query(const AttnArgs& a, const AttnItem& it, int kvh, int qi, int lane) {
  constexpr int DPL = HD / 32;                   // dims per lane
  constexpr int PS = HD + 2;
  using Raw = typename std::conditional<HD == 128, uint2, uint32_t>::type;   // DPL fp16 values
  const int G = a.H / a.KVH;
  const int row = it.row_begin + qi / G, qh = kvh * G + qi % G;
  const DevNode* nd = a.nodes + row;
  const int pos = __ldg(&nd->pos), cend = __ldg(&nd->c_end);
  const int toff = __ldg(&nd->tail_off), ntail = __ldg(&nd->n_tail);
  const int bnd = bulk_end(pos);
  const int nw = pos - bnd + 1;                  // window keys, 1 .. kAttnWindow
  // lane t resolves window key bnd + t: committed cache row, or the branch pool row
  const __half* krow = a.kv_commit;
  const __half* vrow = a.kv_commit;
  if (lane < nw) {
    const int kk = bnd + lane;
    if (kk < cend) {
      krow = a.kv_commit + ((((static_cast<size_t>(it.seq) * a.L + it.layer) * 2) * a.KVH + kvh) * a.max_ctx + kk) * HD;
      vrow = krow + static_cast<size_t>(a.KVH) * a.max_ctx * HD;
    } else {
      const int t = kk - cend;
      int slot = 0;
      if (t < ntail) slot = __ldg(a.tails + toff + t);
      else atomicExch(a.err, DEV_BAD_INDEX);   // cannot happen for a well-formed plan; slot 0 is read
      krow = a.kv_pool + ((((static_cast<size_t>(it.seq) * a.n_slots + slot) * a.L + it.layer) * 2) * a.KVH + kvh) * HD;
      vrow = krow + static_cast<size_t>(a.KVH) * HD;
    }
  }
  float qw[DPL];
  const float* qsrc = a.q + (static_cast<size_t>(row) * a.H + qh) * HD + lane * DPL;
#pragma unroll
  for (int d = 0; d < DPL; ++d) qw[d] = __ldcg(qsrc + d);
  Raw kr[kAttnWindow];
#pragma unroll
  for (int t = 0; t < kAttnWindow; ++t) {
    const __half* kp = reinterpret_cast<const __half*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(krow), t));
    if (t < nw) kr[t] = *reinterpret_cast<const Raw*>(kp + lane * DPL);
  }
  // scores: per key the lane's products in dim order, then the warp butterfly
  float sw[kAttnWindow];
  float mw = -INFINITY;
#pragma unroll
  for (int t = 0; t < kAttnWindow; ++t) {
    sw[t] = -INFINITY;
    if (t < nw) {
      const __half2* h2p = reinterpret_cast<const __half2*>(&kr[t]);
      float dp = 0.0f;
#pragma unroll
      for (int d = 0; d < DPL; d += 2) {
        const float2 f = __half22float2(h2p[d / 2]);
        dp = fmaf(qw[d], f.x, dp);
        dp = fmaf(qw[d + 1], f.y, dp);
      }
      sw[t] = warp_sum(dp) * a.scale_log2;
      mw = fmaxf(mw, sw[t]);
    }
  }
  Raw vr[kAttnWindow];   // value rows after the key rows: fewer registers live at once
#pragma unroll
  for (int t = 0; t < kAttnWindow; ++t) {
    const __half* vp = reinterpret_cast<const __half*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(vrow), t));
    if (t < nw) vr[t] = *reinterpret_cast<const Raw*>(vp + lane * DPL);
  }
  float lw = 0.0f, ow[DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) ow[d] = 0.0f;
#pragma unroll
  for (int t = 0; t < kAttnWindow; ++t) {
    if (t < nw) {
      const float pt = exp2f(sw[t] - mw);
      lw = __fadd_rn(lw, pt);
      const __half2* h2p = reinterpret_cast<const __half2*>(&vr[t]);
#pragma unroll
      for (int d = 0; d < DPL; d += 2) {
        const float2 f = __half22float2(h2p[d / 2]);
        ow[d] = fmaf(pt, f.x, ow[d]);
        ow[d + 1] = fmaf(pt, f.y, ow[d + 1]);
      }
    }
  }
  float* rec = a.part + ((static_cast<size_t>(row) * a.H + qh) * a.part_slots + (a.part_slots - 1)) * PS;
#pragma unroll
  for (int d = 0; d < DPL; ++d) __stcg(rec + lane * DPL + d, ow[d]);
  if (lane == 0) {
    __stcg(rec + HD, mw);
    __stcg(rec + HD + 1, lw);
  }
}

// Final combination of one query: the bulk groups' records in group order, then the window
// record; the output is written as a hi/lo bf16 pair.  The loads of up to 16 groups are
// issued together, before the arithmetic.
template <int HD>
__device__ __forceinline__ void combine_query(const AttnArgs& a, const AttnItem& it, int kvh, int qi, int lane) {
  constexpr int DPL = HD / 32;
  constexpr int PS = HD + 2;
  const int G = a.H / a.KVH;
  const int row = it.row_begin + qi / G, qh = kvh * G + qi % G;
  const float* base = a.part + (static_cast<size_t>(row) * a.H + qh) * a.part_slots * PS;
  const float* wrec = base + (a.part_slots - 1) * PS;
  float mg[2] = {-INFINITY, -INFINITY}, lg[2] = {0.0f, 0.0f};
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int gg = lane + 32 * h2;
    if (gg < it.n_groups) {
      mg[h2] = __ldcg(base + gg * PS + HD);
      lg[h2] = __ldcg(base + gg * PS + HD + 1);
    }
  }
  const float mw = __ldcg(wrec + HD), lw = __ldcg(wrec + HD + 1);
  float ow[DPL], pv[16][DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) ow[d] = __ldcg(wrec + lane * DPL + d);
#pragma unroll
  for (int e = 0; e < 16; ++e)
#pragma unroll
    for (int d = 0; d < DPL; ++d) pv[e][d] = e < it.n_groups ? __ldcg(base + e * PS + lane * DPL + d) : 0.0f;
  const float M = fmaxf(warp_max(fmaxf(mg[0], mg[1])), mw);
  float wg[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) wg[h2] = (lg[h2] > 0.0f) ? exp2f(mg[h2] - M) : 0.0f;
  const float ww = exp2f(mw - M);
  const float L = __fadd_rn(warp_sum(__fadd_rn(lg[0] * wg[0], lg[1] * wg[1])), lw * ww);
  float O[DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) O[d] = 0.0f;
  for (int g16 = 0; g16 < it.n_groups; g16 += 16) {   // groups in order
    if (g16 > 0) {
#pragma unroll
      for (int e = 0; e < 16; ++e)
#pragma unroll
        for (int d = 0; d < DPL; ++d)
          pv[e][d] = g16 + e < it.n_groups ? __ldcg(base + (g16 + e) * PS + lane * DPL + d) : 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int gg = g16 + e;
      const float wv = __shfl_sync(0xffffffffu, gg < 32 ? wg[0] : wg[1], gg & 31);
      if (gg >= it.n_groups || wv == 0.0f) continue;
#pragma unroll
      for (int d = 0; d < DPL; ++d) O[d] = fmaf(wv, pv[e][d], O[d]);
    }
  }
  const float invl = 1.0f / L;
  const size_t lo = static_cast<size_t>(a.plane_rows) * a.H * HD;
#pragma unroll
  for (int d = 0; d < DPL; ++d) {
    const float v = fmaf(ww, ow[d], O[d]) * invl;
    const size_t oo = static_cast<size_t>(row) * a.H * HD + qh * HD + lane * DPL + d;
    store_pair(a.out + oo, a.out + lo + oo, v);
  }
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ AttnArgs a) {
  using SM = AttnSmem<HD>;
  constexpr int S = SM::kStages;
  constexpr int PS = HD + 2;                     // partial record: O[HD], m, l
  constexpr int KS_PER_CHAIN = HD / 16 / 4;      // QK k-steps (16 dims) per accumulator chain
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* red = reinterpret_cast<float*>(smem + SM::oRed);     // [0]: max [16][4], [1]: sum [16][4]
  int* meta = reinterpret_cast<int*>(smem + SM::oMeta);       // bulk bound per pass-local query
  int* qrec = meta + 2 * kQT;                                 // row * H + head of each pass-local query
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::oBar);
  uint64_t* empty = full + S;
  uint64_t* q_full = empty + S;   // query tile written (epilogue -> MMA)
  uint64_t* s_full = q_full + 1;  // scores in TMEM (MMA -> epilogue)
  uint64_t* p_full = s_full + 1;  // probability tile written (epilogue -> MMA)
  uint64_t* o_full = p_full + 1;  // group output in TMEM (MMA -> epilogue)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_full + 1);
  volatile int* sflag = reinterpret_cast<volatile int*>(tmem_slot + 1);   // [1] abort, [2] next combination

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = gridDim.x, cta = blockIdx.x;
  const int u0 = static_cast<int>((static_cast<long long>(cta) * a.n_units) / C);
  const int u1 = static_cast<int>((static_cast<long long>(cta + 1) * a.n_units) / C);
  const int n_my = u1 - u0;
  const int G = a.H / a.KVH;
  unsigned long long* tl = a.timeline ? a.timeline + static_cast<size_t>(cta) * kAttnTimelineSlots : nullptr;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 128);
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(o_full, 1);
    sflag[1] = 0;
    sflag[2] = -1;
    fence_mbar_init();
    tma_prefetch(&tmKV);
  }
  // rows of a tile beyond what TMA writes keep finite values: zero the ring (and the zero
  // atom) once, so a masked key (p = 0) never meets a non-finite value in the MMA
  for (uint32_t o = tid * 16; o < SM::oRed; o += kAttnThreads * 16)
    *reinterpret_cast<uint4*>(smem + o) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // q and this round's K/V come from the preceding launch; the K/V producer of a decode
  // round reads only keys committed in earlier rounds and starts without it
  if (!(warp == 0 && a.early_kv)) griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ---------------- producer: committed K and V tiles of each unit ----------------
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      UnitCursor cu;
      cu.init(a, u0);
      for (int i = 0; i < n_my; ++i, cu.next(a)) {
        const int st = i % S;
        if (i >= S && !mbar_wait(&empty[st], static_cast<uint32_t>((i / S) - 1) & 1u, a.err, DEV_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
        const UnitCursor& ur = cu;
        const AttnItem& it = cu.it;
        const int g0 = ur.g * kAttnGroupPos;
        const int n_com = max(0, min(kAttnGroupPos, bulk_end(it.max_pos) - g0));
        const int nbox = (n_com + kBoxRows - 1) / kBoxRows;
        constexpr int halves = HD / 64;
        mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(2 * nbox * halves * kBoxRows * 128));
        const int row_k = ((((it.seq * a.L + it.layer) * 2 + 0) * a.KVH + ur.kvh) * a.max_ctx) + g0;
        const int row_v = row_k + a.KVH * a.max_ctx;
        uint8_t* sk = ring + static_cast<size_t>(st) * SM::kStage;
        uint8_t* sv = sk + SM::kTile;
        for (int b = 0; b < nbox; ++b) {
#pragma unroll
          for (int h = 0; h < halves; ++h) {
            const uint32_t off = static_cast<uint32_t>(h * kAttnGroupPos * 128 + b * kBoxRows * 128);
            tma_load_2d(sk + off, &tmKV, &full[st], h * 64, row_k + b * kBoxRows);
            tma_load_2d(sv + off, &tmKV, &full[st], h * 64, row_v + b * kBoxRows);
          }
        }
        issued = i + 1;
      }
      if (!ok) {   // drain the copies still in flight before the CTA exits
        for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
          mbar_wait(&full[i % S], static_cast<uint32_t>(i / S) & 1u, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // S = K [Qhi|Qlo]^T and O^T = V^T [Phi|Plo]^T with N = 32 (hi columns 0-15, lo 16-31),
    // each over four independent accumulator chains (a quarter of the dims / keys each) so
    // the chains' MMAs overlap; the epilogue sums chains and halves in a fixed order.
    // This warp also publishes each finished unit to the combining CTA (a gpu-scope release
    // increment of the pair's counter), off the epilogue's path: the epilogue wrote the
    // unit's partials before it posted the next query tile, which this warp waited for; the
    // release is issued after the next pass's QK^T so that MMA does not wait for it.
    if (lane == 0) {
      const uint32_t id_qk = idesc_f16_f32(128, 2 * kQT, false);
      const uint32_t id_pv = idesc_f16_f32(128, 2 * kQT, true);
      const uint32_t d_s = tmem_base, d_o = tmem_base + 4 * 2 * kQT;
      const uint32_t qt = smem_u32(smem + SM::oQ), pt = smem_u32(smem + SM::oP);
      uint32_t np = 0;   // passes so far (barrier phases)
      int* pending = nullptr;   // counter of the unit whose partials the next p_full wait covers
      bool ok = true;
      UnitCursor cu;
      cu.init(a, u0);
      for (int i = 0; i < n_my && ok; ++i, cu.next(a)) {
        const UnitCursor& ur = cu;
        const AttnItem& it = cu.it;
        const int st = i % S;
        const int n_pass = ((it.row_end - it.row_begin) * G + kQT - 1) / kQT;
        const uint32_t kt = smem_u32(ring + static_cast<size_t>(st) * SM::kStage);
        const uint32_t vt = kt + SM::kTile;
        const uint32_t lbo_v = (HD == 128) ? 64u * 256u : smem_u32(smem + SM::oZero) - vt;
        if (!mbar_wait(&full[st], static_cast<uint32_t>(i / S) & 1u, a.err, DEV_TIMEOUT_FULL)) break;
        for (int p = 0; p < n_pass; ++p, ++np) {
          if (!mbar_wait(q_full, np & 1u, a.err, DEV_TIMEOUT_FULL)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int e = 0; e < KS_PER_CHAIN; ++e) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {        // chain c: dims [c HD/4, (c+1) HD/4)
              const int ks = c * KS_PER_CHAIN + e;
              const uint32_t off_a = static_cast<uint32_t>((ks >> 2) * kAttnGroupPos * 128 + (ks & 3) * 32);
              const uint32_t off_b = static_cast<uint32_t>((ks >> 2) * 2 * kQT * 128 + (ks & 3) * 32);
              umma_bf16(d_s + c * 2 * kQT, sw128_kmajor_desc(kt + off_a), sw128_kmajor_desc(qt + off_b), id_qk,
                        e > 0 ? 1u : 0u);
            }
          }
          umma_commit(s_full);
          if (pending) {   // publish the previous unit while this pass's QK^T runs
            asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(pending) : "memory");
            pending = nullptr;
          }
          if (!mbar_wait(p_full, np & 1u, a.err, DEV_TIMEOUT_FULL)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int e = 0; e < 2; ++e) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {        // chain c: keys [32c, 32c + 32)
              const int ks = 2 * c + e;
              const uint64_t ad = sw128_mnmajor_desc(vt + ks * 16 * 128, lbo_v, 1024);
              const uint32_t off_b = static_cast<uint32_t>((ks >> 2) * 2 * kQT * 128 + (ks & 3) * 32);
              umma_bf16(d_o + c * 2 * kQT, ad, sw128_kmajor_desc(pt + off_b), id_pv, e > 0 ? 1u : 0u);
            }
          }
          umma_commit(o_full);
          if (p == n_pass - 1) {
            umma_commit(&empty[st]);   // the stage is free once these MMAs complete
            pending = a.counters + it.counter * a.KVH + ur.kvh;
          }
        }
      }
    }
  } else if (warp < 6) {
    // ---------------- epilogue: query tiles, softmax, partials ----------------
    // Per pass n: scores -> probability tile (post) -> the next pass's query tile (post) ->
    // output -> partial records.  Building the next query tile before the partial stores
    // lets the next QK^T run while the stores drain, and keeps those stores out of the
    // proxy fences.
    const int et = tid - 64;                   // 0..127
    const int lq = warp & 3;                   // TMEM lane quarter of this warp
    const int r = lq * 32 + lane;              // TMEM row: key (scores) or value dim (output)
    const uint32_t t_row = static_cast<uint32_t>(lq * 32) << 16;
    uint8_t* qtile = smem + SM::oQ;
    uint8_t* ptile = smem + SM::oP;
    auto epi_sync = [] { named_bar_sync(kEpiBar, 128); };
    constexpr int QD = HD / 8;                 // query dims per thread (8 threads per query)
    const int qj = et >> 3, qd0 = (et & 7) * QD;
    unsigned long long* etl = (tl && et == 0) ? tl : nullptr;
    // this thread's slice of a pass's queries (fp32) and, for et < 16, the query's
    // position and committed extent -- loaded one pass ahead
    float qv[QD];
    int qpos = -1, qcend = 0;
    auto load_q = [&](const PassCursor& x) {
      const int nq = x.c.n_queries(G);
      const int qi = x.p * kQT + qj;
#pragma unroll
      for (int e = 0; e < QD; ++e) qv[e] = 0.0f;
      if (qi < nq) {
        const int row = x.c.it.row_begin + qi / G, qh = x.c.kvh * G + qi % G;
        const float4* src = reinterpret_cast<const float4*>(a.q + (static_cast<size_t>(row) * a.H + qh) * HD + qd0);
#pragma unroll
        for (int e = 0; e < QD / 4; ++e) {
          const float4 v = __ldcg(src + e);
          qv[4 * e] = v.x; qv[4 * e + 1] = v.y; qv[4 * e + 2] = v.z; qv[4 * e + 3] = v.w;
        }
      }
      qpos = -1;
      qcend = 0;
      const int mi = x.p * kQT + et;
      if (et < kQT && mi < nq) {
        const int row = x.c.it.row_begin + mi / G;
        qpos = __ldg(&a.nodes[row].pos);
        qcend = __ldg(&a.nodes[row].c_end);
      }
    };
    // query tile (hi rows 0-15, lo rows 16-31), bulk bounds and record rows of pass x (buffer b)
    auto post_q = [&](const PassCursor& x, int b) {
#pragma unroll
      for (int e = 0; e < QD; e += 8) {
        __align__(16) __half h8[8], l8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) split_f16(qv[e + k], h8[k], l8[k]);
        *reinterpret_cast<uint4*>(qtile + sw_elem_off(qj, qd0 + e, 2 * kQT)) = *reinterpret_cast<const uint4*>(h8);
        *reinterpret_cast<uint4*>(qtile + sw_elem_off(kQT + qj, qd0 + e, 2 * kQT)) = *reinterpret_cast<const uint4*>(l8);
      }
      if (et < kQT) {
        const int bnd = qpos >= 0 ? bulk_end(qpos) : 0;
        if (bnd > qcend) atomicExch(a.err, DEV_BAD_INDEX);   // a branch key would be in the bulk
        meta[b * kQT + et] = bnd;
        const int qi = x.p * kQT + et;
        qrec[b * kQT + et] = (x.c.it.row_begin + qi / G) * a.H + x.c.kvh * G + qi % G;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    };
    if (etl) {
      etl[0] = global_timer_ns();
      etl[2] = static_cast<unsigned long long>(n_my);
    }
    uint32_t np = 0;
    // cur: the pass being computed; nx: the next (its queries are in registers); nn: the one after
    PassCursor cur, nx, nn;
    bool aborted = false;
    if (n_my > 0) {
      cur.init(a, u0);
      nx = cur;
      nx.next(a, G, n_my);
      nn = nx;
      if (nn.i < n_my) nn.next(a, G, n_my);
      load_q(cur);
      post_q(cur, 0);
      if (nx.i < n_my) load_q(nx);
    }
    while (n_my > 0 && cur.i < n_my && !aborted) {
      const int i = cur.i, p = cur.p;
      const UnitCursor& ur = cur.c;
      const AttnItem& it = cur.c.it;
      const int g0 = ur.g * kAttnGroupPos;
      const int nq = cur.c.n_queries(G);
      const int nb = min(kQT, nq - p * kQT);
      const int b = np & 1;                    // meta / record-row buffer of this pass
      unsigned long long* ut = (etl && i < kAttnTimelineUnits && p == 0) ? etl + 3 + 8 * i : nullptr;
      // (1) scores -> masked exp2 -> probability tile; group max and sum per query
      if (!mbar_wait(s_full, np & 1u, a.err, DEV_TIMEOUT_ACC)) sflag[1] = 1;
      epi_sync();   // this pass's bounds visible; abort visible
      if (sflag[1]) { aborted = true; break; }
      if (ut) ut[1] = global_timer_ns();
      tc_fence_after();
      float s16[kQT];
      tmem_chain_sum(tmem_base + t_row, s16);
      const int key = g0 + r;
      float* rmax = red;
      float* rsum = red + 4 * kQT;
      // the pass's first K >= nb query columns (the probability tile's other columns keep
      // finite values from earlier passes; their outputs are never stored)
      auto softmax = [&](auto kc) {
        constexpr int K = decltype(kc)::value;
        constexpr int LPQ = 32 / K;   // lanes holding one query's reduction
        float s[K];
#pragma unroll
        for (int j = 0; j < K; ++j) s[j] = (j < nb && key < meta[b * kQT + j]) ? s16[j] * a.scale_log2 : -INFINITY;
        {
          const float m = warp_reduce_transposed<K, true>(s, lane);
          if ((lane & (LPQ - 1)) == 0) rmax[(lane / LPQ) * 4 + lq] = m;   // [query][key quarter]
        }
        epi_sync();
#pragma unroll
        for (int j = 0; j < K; ++j) {
          const float4 m4 = *reinterpret_cast<const float4*>(rmax + j * 4);
          const float gmax = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
          s[j] = (s[j] == -INFINITY) ? 0.0f : exp2f(s[j] - gmax);
          __half h, l;
          split_f16(s[j], h, l);
          *reinterpret_cast<__half*>(ptile + sw_elem_off(j, r, 2 * kQT)) = h;
          *reinterpret_cast<__half*>(ptile + sw_elem_off(kQT + j, r, 2 * kQT)) = l;
        }
        const float ps = warp_reduce_transposed<K, false>(s, lane);
        if ((lane & (LPQ - 1)) == 0) rsum[(lane / LPQ) * 4 + lq] = ps;
      };
      if (nb <= 4) softmax(std::integral_constant<int, 4>{});
      else if (nb <= 8) softmax(std::integral_constant<int, 8>{});
      else softmax(std::integral_constant<int, 16>{});
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
      if (ut) ut[2] = global_timer_ns();
      // (2) the next pass's query tile (its queries were loaded one pass ahead), and the
      // loads of the pass after it
      if (nx.i < n_my) {
        post_q(nx, b ^ 1);
        if (nn.i < n_my) load_q(nn);
      }
      if (ut) ut[3] = global_timer_ns();
      // (3) group output -> partial records (O, m, l) of the pass's queries
      if (!mbar_wait(o_full, np & 1u, a.err, DEV_TIMEOUT_ACC)) sflag[1] = 1;
      epi_sync();   // sums visible; abort visible
      if (sflag[1]) { aborted = true; break; }
      if (ut) ut[4] = global_timer_ns();
      tc_fence_after();
      float o[kQT];
      tmem_chain_sum(tmem_base + 4 * 2 * kQT + t_row, o);
      tc_fence_before();
      if (r < HD) {
#pragma unroll
        for (int j = 0; j < kQT; ++j)
          if (j < nb) __stcg(a.part + (static_cast<size_t>(qrec[b * kQT + j]) * a.part_slots + ur.g) * PS + r, o[j]);
      }
      if (et < nb) {   // the query's max and its sum in key-quarter order
        float* pp = a.part + (static_cast<size_t>(qrec[b * kQT + et]) * a.part_slots + ur.g) * PS;
        const float4 m4 = *reinterpret_cast<const float4*>(rmax + et * 4);
        __stcg(pp + HD, fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w)));
        const float4 s4 = *reinterpret_cast<const float4*>(rsum + et * 4);
        __stcg(pp + HD + 1, __fadd_rn(__fadd_rn(s4.x, s4.y), __fadd_rn(s4.z, s4.w)));
      }
      if (ut) ut[5] = global_timer_ns();
      ++np;
      cur = nx;
      nx = nn;
      if (nn.i < n_my) nn.next(a, G, n_my);
    }
    // the last unit's partials are published here (the MMA warp publishes the others)
    epi_sync();
    if (et == 0 && !aborted && n_my > 0) {
      const UnitRef ur = unit_ref(a, u0 + n_my - 1);
      const AttnItem it = a.items[ur.item];
      asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(a.counters + it.counter * a.KVH + ur.kvh)
                   : "memory");
    }
    if (etl) etl[1] = global_timer_ns();
  } else {
    // ---------------- merge warps: window parts and final combinations ----------------
    // The CTA that owns the last group of an (item, KV head) combines it.  Its window part
    // needs nothing from the other units, so it is computed first, while the units run;
    // the combination waits until all of the pair's units have counted themselves done.
    const int mw = warp - 6;
    UnitCursor cu;
    if (n_my > 0) cu.init(a, u0);
    for (int i = 0; i < n_my; ++i, cu.next(a)) {
      const UnitCursor& ur = cu;
      const AttnItem& it = cu.it;
      if (ur.g != it.n_groups - 1) continue;
      const int nq = (it.row_end - it.row_begin) * G;
      for (int qi = mw; qi < nq; qi += kMergeWarps) window_query<HD>(a, it, ur.kvh, qi, lane);
    }
    // the combinations, in the order the pairs complete: sweep the owned pairs, combine
    // every one whose units have all counted themselves done
    // (a combined pair's counter is reset to 0, so a later sweep never picks it again)
    int n_merge = 0;
    int remaining = 0;
    if (n_my > 0) cu.init(a, u0);
    for (int i = 0; i < n_my; ++i, cu.next(a))
      if (cu.g == cu.it.n_groups - 1) ++remaining;
    const uint64_t t_start = global_timer_ns();
    volatile int* flag = sflag + 2;   // [2]: index of the next pair to combine (-1: none ready)
    while (remaining > 0) {
      if (tid == 6 * 32) {
        int pick = -1;
        UnitCursor c2;
        c2.init(a, u0);
        for (int i = 0; i < n_my && pick < 0; ++i, c2.next(a)) {
          if (c2.g != c2.it.n_groups - 1) continue;
          int v;
          asm volatile("ld.acquire.gpu.global.s32 %0, [%1];"
                       : "=r"(v)
                       : "l"(a.counters + c2.it.counter * a.KVH + c2.kvh)
                       : "memory");
          if (v >= c2.it.n_groups) pick = i;
        }
        if (pick < 0 && global_timer_ns() - t_start > kWaitLimitNs) {
          atomicExch(a.err, DEV_TIMEOUT_ACC);
          pick = -2;
        }
        *flag = pick;
        if (pick == -1) __nanosleep(128);
      }
      named_bar_sync(kMergeBar, 32 * kMergeWarps);
      const int pick = *flag;
      named_bar_sync(kMergeBar, 32 * kMergeWarps);   // everyone read the pick before it changes
      if (pick == -2) break;
      if (pick < 0) continue;
      UnitCursor c3;
      c3.init(a, u0 + pick);
      unsigned long long* mt = (tl && tid == 6 * 32 && n_merge < 4) ? tl + 3 + 8 * kAttnTimelineUnits + 2 * n_merge
                                                                     : nullptr;
      if (mt) mt[0] = global_timer_ns();
      const int nq = (c3.it.row_end - c3.it.row_begin) * G;
      for (int qi = mw; qi < nq; qi += kMergeWarps) combine_query<HD>(a, c3.it, c3.kvh, qi, lane);
      named_bar_sync(kMergeBar, 32 * kMergeWarps);
      if (tid == 6 * 32) {
        a.counters[c3.it.counter * a.KVH + c3.kvh] = 0;   // ready for the next launch
        if (mt) mt[1] = global_timer_ns();
      }
      ++n_merge;
      --remaining;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
}

template <int HD>
static cudaError_t launch_attn_hd(cudaLaunchConfig_t cfg, const CUtensorMap& tm, const AttnArgs& a) {
  static bool set = false;
  cfg.dynamicSmemBytes = AttnSmem<HD>::kTotal;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cfg.dynamicSmemBytes));
    if (e == cudaSuccess) e = apply_carveout(attn_kernel<HD>);
    if (e != cudaSuccess) return e;
    set = true;
  }
  return cudaLaunchKernelEx(&cfg, attn_kernel<HD>, tm, a);
}

cudaError_t launch_attention(const CUtensorMap& tm, const AttnArgs& a, int n_ctas, cudaStream_t st, bool pdl) {
  if (a.n_items <= 0 || a.n_units <= 0) return cudaSuccess;
  if (!a.nodes || !a.items || !a.tails || !a.q || !a.kv_commit || !a.kv_pool || !a.out || !a.part || !a.counters ||
      !a.err || a.plane_rows < 1 || a.part_slots < 2 || a.part_slots > kAttnMaxGroups + 1 || n_ctas < 1 ||
      (a.hd != 64 && a.hd != 128))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_ctas < a.n_units ? n_ctas : a.n_units));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.hd == 128) return launch_attn_hd<128>(cfg, tm, a);
  return launch_attn_hd<64>(cfg, tm, a);
}

// ============================================================================================
// Prefill: causal attention of a pass of consecutive prompt positions, flash-attention style
// on the tensor cores.  A CTA takes 128 query rows (128 / G positions x the G query heads of
// one KV head) against every key position up to its last row's, in 128-key tiles streamed
// by TMA from the committed cache:
//   S = [Qhi|Qlo] K^T      (M = 128 query rows, N = 128 keys; Q as an fp16 hi/lo pair)
//   O += P V               (M = 128 query rows, N = head_dim; P fp16, V an MN-major operand)
// One thread per query row reads its row of S from TMEM, so the softmax needs no exchange
// between threads.  Two passes: the first takes each row's maximum over all its keys (from
// Qhi alone -- any value near the maximum keeps the exponentials in range), the second
// forms P = exp2(s - max) and accumulates O and the row sums, so O never needs rescaling.
// Prefill numerics are shared by DEX and AR decoding, so they need not match a decode
// round's bits.
// ============================================================================================
namespace {
constexpr int kPfThreads = 192;   // producer, MMA issuer, four softmax warps
constexpr int kPfStages = 2;

template <int HD>
struct PfSmem {
  static constexpr uint32_t kTile = 128 * HD * 2;            // [128 rows][HD] fp16, HD/64 atoms of 16 KB
  static constexpr uint32_t oQhi = 0, oQlo = kTile;
  static constexpr uint32_t oP = 2 * kTile;                  // [128 rows][128 keys] fp16
  static constexpr uint32_t oRing = oP + 128 * 128 * 2;      // stages of K then V
  static constexpr uint32_t kStage = 2 * kTile;
  static constexpr uint32_t oBar = oRing + kPfStages * kStage;
  static constexpr uint32_t kTotal = oBar + (2 * kPfStages + 8) * 8 + 16 + 1024;
};
static_assert(PfSmem<128>::kTotal <= 227 * 1024, "prefill attention shared memory");

__host__ __device__ constexpr uint32_t idesc_f16_f32_bmn(int M, int N) {   // A K-major, B MN-major
  return (1u << 4) | (1u << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
}  // namespace

template <int HD>
__global__ void __launch_bounds__(kPfThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ PrefillAttnArgs a) {
  using SM = PfSmem<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::oBar);
  uint64_t* empty = full + kPfStages;
  uint64_t* s_full = empty + kPfStages;   // [2] scores of a tile in S[b]
  uint64_t* s_free = s_full + 2;          // [2] S[b] read by every row
  uint64_t* q_full = s_free + 2;          // query tiles written
  uint64_t* p_full = q_full + 1;          // probability tile written
  uint64_t* p_free = p_full + 1;          // probability tile consumed by its PV
  uint64_t* o_full = p_free + 1;          // every PV complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_full + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.H / a.KVH, QP = 128 / G;   // query heads per KV head, positions per block
  const int kvh = blockIdx.y;
  const int p0 = blockIdx.x * QP;            // first node row (position index) of the block
  const int np = min(QP, a.n_rows - p0);     // positions in the block
  if (np <= 0) return;
  const int max_pos = __ldg(&a.nodes[p0 + np - 1].pos);
  const int nkt = max_pos / 128 + 1;         // key tiles 0 .. nkt-1

  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 128);
    }
    mbar_init(q_full, 128);
    mbar_init(p_full, 128);
    mbar_init(p_free, 1);
    mbar_init(o_full, 1);
    fence_mbar_init();
    tma_prefetch(&tmKV);
  }
  // key rows past a tile's last loaded row keep finite values: zero the ring once
  for (uint32_t o = SM::oRing + tid * 16; o < SM::oBar; o += kPfThreads * 16)
    *reinterpret_cast<uint4*>(smem + o) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);   // S[0], S[1]: 128 columns each; O: HD columns
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t t_s0 = tmem_base, t_o = tmem_base + 256;
  griddep_wait();   // q and the pass's K/V come from the preceding launches
  griddep_launch_dependents();

  constexpr int KS = HD / 16;   // 16-dim k steps of QK^T
  if (warp == 0) {
    // ---------------- producer: K tiles (pass 1), then K and V tiles (pass 2) ----------------
    if (lane == 0) {
      const int row_k = (((a.seq * a.L + a.layer) * 2 + 0) * a.KVH + kvh) * a.max_ctx;
      const int row_v = row_k + a.KVH * a.max_ctx;
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < 2 * nkt && ok; ++j) {
        const int kt = j < nkt ? j : j - nkt;
        const bool with_v = j >= nkt;
        const int st = j % kPfStages;
        if (j >= kPfStages &&
            !mbar_wait(&empty[st], static_cast<uint32_t>((j / kPfStages) - 1) & 1u, a.err, DEV_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
        const int nk = min(128, max_pos + 1 - kt * 128);   // keys of the tile any row can see
        const int nbox = (nk + 31) / 32;
        constexpr int halves = HD / 64;
        mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>((with_v ? 2 : 1) * nbox * halves * 32 * 128));
        uint8_t* sk = smem + SM::oRing + static_cast<size_t>(st) * SM::kStage;
        for (int bx = 0; bx < nbox; ++bx) {
#pragma unroll
          for (int h = 0; h < halves; ++h) {
            const uint32_t off = static_cast<uint32_t>(h * 128 * 128 + bx * 32 * 128);
            tma_load_2d(sk + off, &tmKV, &full[st], h * 64, row_k + kt * 128 + bx * 32);
            if (with_v) tma_load_2d(sk + SM::kTile + off, &tmKV, &full[st], h * 64, row_v + kt * 128 + bx * 32);
          }
        }
        issued = j + 1;
      }
      if (!ok) {
        for (int j = (issued > kPfStages ? issued - kPfStages : 0); j < issued; ++j)
          mbar_wait(&full[j % kPfStages], static_cast<uint32_t>(j / kPfStages) & 1u, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_qk = idesc_f16_f32(128, 128, false);
      const uint32_t id_pv = idesc_f16_f32_bmn(128, HD);
      const uint32_t qhi = smem_u32(smem + SM::oQhi), qlo = smem_u32(smem + SM::oQlo);
      const uint32_t pt = smem_u32(smem + SM::oP);
      bool ok = mbar_wait(q_full, 0u, a.err, DEV_TIMEOUT_FULL);
      for (int j = 0; j < 2 * nkt && ok; ++j) {
        const bool pass2 = j >= nkt;
        const int kt = pass2 ? j - nkt : j;
        const int st = j % kPfStages, b = j & 1;
        if (!mbar_wait(&full[st], static_cast<uint32_t>(j / kPfStages) & 1u, a.err, DEV_TIMEOUT_FULL)) break;
        if (j >= 2 && !mbar_wait(&s_free[b], static_cast<uint32_t>((j >> 1) - 1) & 1u, a.err, DEV_TIMEOUT_ACC)) break;
        tc_fence_after();
        const uint32_t kt_s = smem_u32(smem + SM::oRing + static_cast<size_t>(st) * SM::kStage);
        const uint32_t d_s = t_s0 + static_cast<uint32_t>(b) * 128;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t off = static_cast<uint32_t>((ks >> 2) * 128 * 128 + (ks & 3) * 32);
          const uint64_t kdesc = sw128_kmajor_desc(kt_s + off);
          umma_bf16(d_s, sw128_kmajor_desc(qhi + off), kdesc, id_qk, ks > 0 ? 1u : 0u);
          if (pass2) umma_bf16(d_s, sw128_kmajor_desc(qlo + off), kdesc, id_qk, 1u);
        }
        umma_commit(&s_full[b]);
        if (!pass2) {
          umma_commit(&empty[st]);
          continue;
        }
        if (!mbar_wait(p_full, static_cast<uint32_t>(kt) & 1u, a.err, DEV_TIMEOUT_FULL)) break;
        tc_fence_after();
        const uint32_t vt = kt_s + SM::kTile;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {   // 16 keys per step
          const uint32_t off_p = static_cast<uint32_t>((ks >> 2) * 128 * 128 + (ks & 3) * 32);
          umma_bf16(t_o, sw128_kmajor_desc(pt + off_p), sw128_mnmajor_desc(vt + ks * 16 * 128, 128 * 128, 1024),
                    id_pv, (kt > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(p_free);
        umma_commit(&empty[st]);
      }
      umma_commit(o_full);
    }
  } else {
    // ---------------- softmax: one query row per thread ----------------
    const int lq = warp & 3;
    const int r = lq * 32 + lane;                        // query row = TMEM lane
    const uint32_t t_row = static_cast<uint32_t>(lq * 32) << 16;
    const int pj = r / G, hq = kvh * G + r % G;          // position index in the block, query head
    const bool valid = pj < np;
    const int node = p0 + pj;
    const int pos = valid ? __ldg(&a.nodes[node].pos) : -1;
    // query tiles: fp16 hi/lo pair of the row's query
    {
      const float4* qs = reinterpret_cast<const float4*>(a.q + (static_cast<size_t>(node) * a.H + hq) * HD);
#pragma unroll 4
      for (int e = 0; e < HD; e += 8) {
        __align__(16) __half h8[8], l8[8];
        const float4 x0 = valid ? __ldcg(qs + e / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 x1 = valid ? __ldcg(qs + e / 4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) split_f16(xs[k], h8[k], l8[k]);
        *reinterpret_cast<uint4*>(smem + SM::oQhi + sw_elem_off(r, e, 128)) = *reinterpret_cast<const uint4*>(h8);
        *reinterpret_cast<uint4*>(smem + SM::oQlo + sw_elem_off(r, e, 128)) = *reinterpret_cast<const uint4*>(l8);
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < 2 * nkt && ok; ++j) {
      const bool pass2 = j >= nkt;
      const int kt = pass2 ? j - nkt : j;
      const int b = j & 1;
      if (!mbar_wait(&s_full[b], static_cast<uint32_t>(j >> 1) & 1u, a.err, DEV_TIMEOUT_ACC)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = t_s0 + static_cast<uint32_t>(b) * 128 + t_row;
      const int k0 = kt * 128;
      if (!pass2) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32_nowait(taddr + static_cast<uint32_t>(c * 32), v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (k0 + c * 32 + i <= pos) m = fmaxf(m, __uint_as_float(v[i]) * a.scale_log2);
        }
        tc_fence_before();
        mbar_arrive(&s_free[b]);
        continue;
      }
      // pass 2: P = exp2(s - m) for this tile's keys, the row sum over the fp16 values used
      if (kt > 0 && !mbar_wait(p_free, static_cast<uint32_t>(kt - 1) & 1u, a.err, DEV_TIMEOUT_ACC)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32_nowait(taddr + static_cast<uint32_t>(c * 32), v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          __align__(16) __half p8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int key = k0 + c * 32 + e + k;
            const float pf = (key <= pos) ? exp2f(__uint_as_float(v[e + k]) * a.scale_log2 - m) : 0.0f;
            p8[k] = __float2half_rn(pf);
            l = __fadd_rn(l, __half2float(p8[k]));
          }
          *reinterpret_cast<uint4*>(smem + SM::oP + sw_elem_off(r, c * 32 + e, 128)) =
              *reinterpret_cast<const uint4*>(p8);
        }
      }
      tc_fence_before();
      mbar_arrive(&s_free[b]);
      fence_proxy_async_smem();
      mbar_arrive(p_full);
    }
    // output row: O / l as a bf16 hi/lo pair
    if (ok && mbar_wait(o_full, 0u, a.err, DEV_TIMEOUT_ACC)) {
      tc_fence_after();
      const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
      const size_t lo = static_cast<size_t>(a.plane_rows) * a.H * HD;
      const size_t o0 = (static_cast<size_t>(node) * a.H + hq) * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t v[32];
        tmem_ld32_nowait(t_o + t_row + static_cast<uint32_t>(c * 32), v);
        tmem_wait_ld();
        if (valid) {   // the row's bf16 hi/lo pairs, eight values per 16-byte store
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            __align__(16) __nv_bfloat16 h8[8], l8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float x = __uint_as_float(v[i + k]) * inv;
              h8[k] = __float2bfloat16_rn(x);
              l8[k] = __float2bfloat16_rn(__fsub_rn(x, __bfloat162float(h8[k])));
            }
            *reinterpret_cast<uint4*>(a.out + o0 + c * 32 + i) = *reinterpret_cast<const uint4*>(h8);
            *reinterpret_cast<uint4*>(a.out + lo + o0 + c * 32 + i) = *reinterpret_cast<const uint4*>(l8);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

bool prefill_attention_supported(int H, int KVH, int hd) {
  return (hd == 64 || hd == 128) && KVH > 0 && H % KVH == 0 && 128 % (H / KVH) == 0;
}

template <int HD>
static cudaError_t launch_prefill_hd(cudaLaunchConfig_t cfg, const CUtensorMap& tm, const PrefillAttnArgs& a) {
  static bool set = false;
  cfg.dynamicSmemBytes = PfSmem<HD>::kTotal;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cfg.dynamicSmemBytes));
    if (e == cudaSuccess) e = apply_carveout(attn_prefill_kernel<HD>);
    if (e != cudaSuccess) return e;
    set = true;
  }
  return cudaLaunchKernelEx(&cfg, attn_prefill_kernel<HD>, tm, a);
}

cudaError_t launch_prefill_attention(const CUtensorMap& tm, const PrefillAttnArgs& a, cudaStream_t st, bool pdl) {
  if (a.n_rows <= 0) return cudaSuccess;
  if (!a.nodes || !a.q || !a.out || !a.err || a.plane_rows < a.n_rows || !prefill_attention_supported(a.H, a.KVH, a.hd))
    return cudaErrorInvalidValue;
  const int QP = 128 / (a.H / a.KVH);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((a.n_rows + QP - 1) / QP), static_cast<unsigned>(a.KVH));
  cfg.blockDim = dim3(kPfThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.hd == 128) return launch_prefill_hd<128>(cfg, tm, a);
  return launch_prefill_hd<64>(cfg, tm, a);
}

}  // namespace dex

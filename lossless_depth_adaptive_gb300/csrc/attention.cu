// Lattice-masked attention for the node batches of a DEX round (and prefill chunks).
//
// A node at input position p attends keys 0..p of its own token prefix (section 3.2:
// "ancestry, KV entries, and attention masks" follow the binary lattice).  Keys at
// positions < c_end come from the committed cache (shared by every node of the
// sequence); keys at c_end..p are the branch entries of the node's P-ancestors' slot
// chains and its own, read from the branch pool through the node's tail table.
//
// Work: a unit is (item, KV head, 128-position key group); an item is one sequence's
// contiguous node rows of one layer.  Persistent CTAs (one per SM) take contiguous ranges
// of units.  Warp 0 streams each unit's committed key and value tiles (fp16, up to 128
// rows) into a ring of shared-memory stages with TMA (128-byte swizzle, 32-row boxes, so
// a ragged last group moves only the rows it has); eight consumer warps work on the
// oldest landed stage while the next stages load.  The consumers form two quads; each
// quad takes half of the unit's queries, and within a quad warp w owns keys 32w..32w+31
// of the group.  Scores take lane = key (the swizzle puts the 16-byte chunk c of the
// eight rows a quarter-warp reads in eight distinct bank groups; the query chunk is one
// broadcast read); values take lane = four (or two) output dims, so a warp reads one
// whole value row per load.  A committed key is read from HBM once per (item, KV head).
//
// The arithmetic for a query is fixed by absolute positions only -- 32-key slices aligned
// to position 0, each score summed in chunk order wherever the key row lives (tile or
// pool), slices combined in order within a group, groups combined in group order by the
// unit that finishes an (item, KV head) last -- so a node's output is bit-identical
// whether its keys sit in the committed cache or the branch pool and whatever batch,
// launch or CTA it is computed in.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace dex {

constexpr int kSlices = kAttnGroupPos / 32;           // 32-key slices per group
constexpr int kTeamWarps = 2 * kSlices;               // two quads of consumer warps
constexpr int kAttnThreads = 32 * (1 + kTeamWarps);   // + the producer warp
constexpr int kBoxRows = 32;                          // TMA box height
constexpr int kTeamBar = 1, kQuadBar0 = 2;            // named barriers (ids)
static_assert(kAttnGroupPos == 128 && kSlices == 4, "four 32-key slices per 128-position group");

// Shared-memory plan of a CTA: ring stages (K tile, V tile), two query buffers, the slice
// records of one pass, barriers.
template <int HD, int QB>
struct AttnSmem {
  static constexpr uint32_t kTile = kAttnGroupPos * HD * 2;     // fp16 tile, 1024-aligned
  static constexpr uint32_t kStage = 2 * kTile;
  static constexpr int kStages = (HD == 128) ? 3 : 6;
  static constexpr uint32_t kRing = kStages * kStage;
  static constexpr uint32_t kQ = 2u * QB * HD * 4;              // double-buffered fp32 queries
  static constexpr uint32_t kRec = static_cast<uint32_t>(QB) * kSlices * (HD + 2) * 4;
  static constexpr uint32_t kBars = 2 * kStages * 8 + 16;
  static constexpr uint32_t kTotal = kRing + kQ + kRec + kBars + 1024;   // + alignment slack
};

// q . k over 8-dim chunks in order: four partial sums by feature residue mod 4 (features
// 4c + r go to sum r), two per packed FMA (each element rounded as fmaf), then
// (s0 + s1) + (s2 + s3).
__device__ __forceinline__ void dot8(float2& s01, float2& s23, const float* q, const uint4& kraw) {
  const float4 qa = *reinterpret_cast<const float4*>(q);
  const float4 qb = *reinterpret_cast<const float4*>(q + 4);
  const float2 k0 = __half22float2(*reinterpret_cast<const __half2*>(&kraw.x));
  const float2 k1 = __half22float2(*reinterpret_cast<const __half2*>(&kraw.y));
  const float2 k2 = __half22float2(*reinterpret_cast<const __half2*>(&kraw.z));
  const float2 k3 = __half22float2(*reinterpret_cast<const __half2*>(&kraw.w));
  s01 = __ffma2_rn(make_float2(qa.x, qa.y), k0, s01);
  s23 = __ffma2_rn(make_float2(qa.z, qa.w), k1, s23);
  s01 = __ffma2_rn(make_float2(qb.x, qb.y), k2, s01);
  s23 = __ffma2_rn(make_float2(qb.z, qb.w), k3, s23);
}
__device__ __forceinline__ float dot_finish(const float2& s01, const float2& s23) {
  return __fadd_rn(__fadd_rn(s01.x, s01.y), __fadd_rn(s23.x, s23.y));
}

// 16-byte chunk c (dims 8c..8c+7) of row r of a swizzled fp16 tile: 64-dim halves of
// kAttnGroupPos rows x 128 bytes; chunk cc of row r sits at (cc ^ (r & 7)) * 16.
__device__ __forceinline__ uint32_t tile_chunk_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (kAttnGroupPos * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Dims [lane * DPL, lane * DPL + DPL) of row r of a value tile (or a pool row) as floats.
template <int HD>
__device__ __forceinline__ void value_dims_tile(const uint8_t* tile, int r, int lane, float (&v)[HD / 32]) {
  if constexpr (HD == 128) {   // four dims = 8 bytes: chunk lane / 2, half (lane & 1)
    const uint2 raw =
        *reinterpret_cast<const uint2*>(tile + tile_chunk_off(r, lane >> 1) + ((lane & 1) << 3));
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  } else {                     // two dims = 4 bytes: chunk lane / 4, quarter (lane & 3)
    const uint32_t raw = *reinterpret_cast<const uint32_t*>(tile + tile_chunk_off(r, lane >> 2) + ((lane & 3) << 2));
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw));
    v[0] = a.x; v[1] = a.y;
  }
}
template <int HD>
__device__ __forceinline__ void value_dims_row(const __half* row, int lane, float (&v)[HD / 32]) {
  if constexpr (HD == 128) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(row) + lane);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  } else {
    const uint32_t raw = __ldg(reinterpret_cast<const uint32_t*>(row) + lane);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw));
    v[0] = a.x; v[1] = a.y;
  }
}

// acc[i] += p * v[i] over the lane's output dims, two dims per packed FMA.
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
// Committed rows of group g that some query of the item reads: [g0, g0 + n).
__device__ __forceinline__ int committed_rows(const AttnItem& it, int g) {
  return max(0, min(kAttnGroupPos, min(it.max_cend, it.max_pos + 1) - g * kAttnGroupPos));
}

template <int HD, int QB>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ AttnArgs a) {
  using SM = AttnSmem<HD, QB>;
  constexpr int S = SM::kStages;
  constexpr int DPL = HD / 32;                  // output dims per lane
  constexpr int NCH = HD / 8;                   // 16-byte chunks per fp16 row
  constexpr int QH = QB >= 2 ? QB / 2 : 1;      // queries per quad per pass
  constexpr int PS = HD + 2;                    // slice record: acc[HD], m, l
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* sQ = reinterpret_cast<float*>(smem + SM::kRing);           // [2][QB][HD]
  float* sRec = sQ + 2 * QB * HD;                                   // [QB][kSlices][PS]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kRing + SM::kQ + SM::kRec);
  uint64_t* empty = full + S;
  volatile int* sflag = reinterpret_cast<volatile int*>(empty + S);   // [0] last arriver, [1] abort

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = gridDim.x, cta = blockIdx.x;
  const int u0 = static_cast<int>((static_cast<long long>(cta) * a.n_units) / C);
  const int u1 = static_cast<int>((static_cast<long long>(cta + 1) * a.n_units) / C);
  const int n_my = u1 - u0;
  const int G = a.H / a.KVH;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTeamWarps);
    }
    sflag[0] = 0;
    sflag[1] = 0;
    fence_mbar_init();
    tma_prefetch(&tmKV);
  }
  __syncthreads();
  griddep_wait();   // q and this round's K/V come from the preceding launch
  griddep_launch_dependents();
  if (n_my <= 0) return;

  if (warp == 0) {
    // ---------------- producer: committed K and V tiles of each unit ----------------
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < n_my; ++i) {
        const int st = i % S;
        if (i >= S && !mbar_wait(&empty[st], static_cast<uint32_t>((i / S) - 1) & 1u, a.err, DEV_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
        const UnitRef ur = unit_ref(a, u0 + i);
        const AttnItem it = a.items[ur.item];
        const int n_com = committed_rows(it, ur.g);
        const int nbox = (n_com + kBoxRows - 1) / kBoxRows;
        constexpr int halves = HD / 64;
        mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(2 * nbox * halves * kBoxRows * 128));
        const int row_k = ((((it.seq * a.L + it.layer) * 2 + 0) * a.KVH + ur.kvh) * a.max_ctx) +
                          ur.g * kAttnGroupPos;
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
    return;
  }

  // ---------------- consumers: warps 1..8, quads of four key slices ----------------
  const int cw = warp - 1, quad = cw >> 2, w = cw & 3;
  const int tt = tid - 32;                      // team thread 0..255
  const int qbar = kQuadBar0 + quad;
  auto team_sync = [] { named_bar_sync(kTeamBar, 32 * kTeamWarps); };
  auto quad_sync = [&] { named_bar_sync(qbar, 32 * kSlices); };

  // query pass sequence of this CTA: (unit i, pass p); the next pass's queries are copied
  // into the other buffer while the current one is computed
  auto issue_q = [&](int i, int p, int buf) {
    const UnitRef ur = unit_ref(a, u0 + i);
    const AttnItem it = a.items[ur.item];
    const int nq = (it.row_end - it.row_begin) * G;
    const int q0 = p * QB;
    float* dst = sQ + buf * QB * HD;
    for (int idx = tt * 4; idx < QB * HD; idx += 32 * kTeamWarps * 4) {
      const int j = idx / HD, d = idx - j * HD;
      const int qi = q0 + j;
      if (qi < nq) {
        const int row = it.row_begin + qi / G, qh = ur.kvh * G + qi % G;
        cp_async_16(smem_u32(dst + idx), a.q + (static_cast<size_t>(row) * a.H + qh) * HD + d);
      } else {
        *reinterpret_cast<float4*>(dst + idx) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    cp_async_commit();
  };
  int buf = 0;
  issue_q(0, 0, 0);
  for (int i = 0; i < n_my; ++i) {
    const UnitRef ur = unit_ref(a, u0 + i);
    const AttnItem it = a.items[ur.item];
    const int st = i % S;
    const int g0 = ur.g * kAttnGroupPos;
    const int nq = (it.row_end - it.row_begin) * G;
    const int n_pass = (nq + QB - 1) / QB;
    const uint8_t* sk = ring + static_cast<size_t>(st) * SM::kStage;
    const uint8_t* sv = sk + SM::kTile;
    const bool landed = mbar_wait(&full[st], static_cast<uint32_t>(i / S) & 1u, a.err, DEV_TIMEOUT_FULL);
    if (!landed) sflag[1] = 1;
    const __half* kcom_pool = reinterpret_cast<const __half*>(a.kv_pool);
    // the branch-pool row of key kk (kk >= c_end) of node row nrow
    auto pool_row = [&](int nrow, int kk, int kv) -> const __half* {
      const DevNode* nd = a.nodes + nrow;
      const int t = kk - nd->c_end;
      int slot = 0;
      if (t >= 0 && t < nd->n_tail) {
        slot = a.tails[nd->tail_off + t];
      } else {   // cannot happen for a well-formed plan; reported, and slot 0 is read instead
        atomicExch(a.err, DEV_BAD_INDEX);
      }
      return kcom_pool +
             ((((static_cast<size_t>(it.seq) * a.n_slots + slot) * a.L + it.layer) * 2 + kv) * a.KVH + ur.kvh) * HD;
    };
    for (int p = 0; p < n_pass; ++p) {
      cp_async_wait_all();   // this pass's queries (copied while the previous pass ran)
      team_sync();           // ... visible to all; every thread is done with the other buffer
      if (sflag[1]) break;
      // the next pass's queries into the other buffer, overlapping this pass
      if (p + 1 < n_pass) issue_q(i, p + 1, buf ^ 1);
      else if (i + 1 < n_my) issue_q(i + 1, 0, buf ^ 1);
      const float* qbuf = sQ + buf * QB * HD;
      const int q0 = p * QB;
      const int nb = min(QB, nq - q0);
      // this quad's queries: pass-local slots jb .. jb + QH - 1
      const int jb = quad * QH;
      int pos[QH], cend[QH], nrow[QH];
      int cmin = 0x7fffffff, pmax = -1;
#pragma unroll
      for (int j = 0; j < QH; ++j) {
        pos[j] = -1;
        cend[j] = 0;
        nrow[j] = it.row_begin;
        if (jb + j < nb) {
          nrow[j] = it.row_begin + (q0 + jb + j) / G;
          pos[j] = __ldg(&a.nodes[nrow[j]].pos);
          cend[j] = __ldg(&a.nodes[nrow[j]].c_end);
          cmin = min(cmin, cend[j]);
          pmax = max(pmax, pos[j]);
        }
      }
      const bool quad_live = jb < nb;
      const int kr = 32 * w + lane;             // this lane's key row within the group
      const int k = g0 + kr;
      float sc[QH];
      if (quad_live && k < cmin && k <= pmax) {   // committed for every query of the quad
        float2 s01[QH], s23[QH];
#pragma unroll
        for (int j = 0; j < QH; ++j) s01[j] = s23[j] = make_float2(0.0f, 0.0f);
#pragma unroll 4
        for (int c = 0; c < NCH; ++c) {
          const uint4 kraw = *reinterpret_cast<const uint4*>(sk + tile_chunk_off(kr, c));
#pragma unroll
          for (int j = 0; j < QH; ++j)
            if (jb + j < nb) dot8(s01[j], s23[j], qbuf + (jb + j) * HD + 8 * c, kraw);
        }
#pragma unroll
        for (int j = 0; j < QH; ++j)
          sc[j] = (jb + j < nb && k <= pos[j]) ? dot_finish(s01[j], s23[j]) * a.scale_log2 : -INFINITY;
      } else {
#pragma unroll
        for (int j = 0; j < QH; ++j) {
          sc[j] = -INFINITY;
          if (jb + j < nb && k <= pos[j]) {
            float2 s01 = make_float2(0.0f, 0.0f), s23 = make_float2(0.0f, 0.0f);
            if (k < cend[j]) {
              for (int c = 0; c < NCH; ++c)
                dot8(s01, s23, qbuf + (jb + j) * HD + 8 * c, *reinterpret_cast<const uint4*>(sk + tile_chunk_off(kr, c)));
            } else {
              const uint4* prow = reinterpret_cast<const uint4*>(pool_row(nrow[j], k, 0));
              for (int c = 0; c < NCH; ++c) dot8(s01, s23, qbuf + (jb + j) * HD + 8 * c, __ldg(prow + c));
            }
            sc[j] = dot_finish(s01, s23) * a.scale_log2;
          }
        }
      }
      // slice softmax statistics and the value accumulation, keys in order
      float mx[QH], lsum[QH], pr[QH], acc[QH][DPL];
#pragma unroll
      for (int j = 0; j < QH; ++j) {
        mx[j] = warp_max(sc[j]);
        pr[j] = 0.0f;
        lsum[j] = 0.0f;
        if (mx[j] != -INFINITY) {
          pr[j] = exp2f(sc[j] - mx[j]);
          lsum[j] = warp_sum(pr[j]);
        }
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[j][d] = 0.0f;
      }
      if (quad_live) {
        const int ks = g0 + 32 * w;
        const int n_keys = min(32, pmax - ks + 1);   // keys of the slice some query attends
#pragma unroll 2
        for (int u = 0; u < n_keys; ++u) {
          const int key = ks + u;
          if (key < cmin) {   // committed for every query: one row read
            float vv[DPL];
            value_dims_tile<HD>(sv, 32 * w + u, lane, vv);
#pragma unroll
            for (int j = 0; j < QH; ++j) {
              if (jb + j < nb && key <= pos[j]) axpy_dims<DPL>(acc[j], __shfl_sync(0xffffffffu, pr[j], u), vv);
            }
          } else {
#pragma unroll
            for (int j = 0; j < QH; ++j) {
              if (jb + j < nb && key <= pos[j]) {
                float vv[DPL];
                if (key < cend[j]) value_dims_tile<HD>(sv, 32 * w + u, lane, vv);
                else value_dims_row<HD>(pool_row(nrow[j], key, 1), lane, vv);
                axpy_dims<DPL>(acc[j], __shfl_sync(0xffffffffu, pr[j], u), vv);
              }
            }
          }
        }
      }
      // the stage is free once the last pass has read its values
      if (p == n_pass - 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      // slice records of the quad's queries, then the in-order combination of the slices
#pragma unroll
      for (int j = 0; j < QH; ++j) {
        if (jb + j < nb) {
          float* rec = sRec + ((jb + j) * kSlices + w) * PS;
#pragma unroll
          for (int d = 0; d < DPL; ++d) rec[lane * DPL + d] = acc[j][d];
          if (lane == 0) {
            rec[HD] = mx[j];
            rec[HD + 1] = lsum[j];
          }
        }
      }
      quad_sync();
      for (int j = jb + w; j < min(nb, jb + QH); j += kSlices) {
        const int qi = q0 + j;
        const int row = it.row_begin + qi / G, qh = ur.kvh * G + qi % G;
        const float* r0 = sRec + (j * kSlices) * PS;
        float mw[kSlices], wgt[kSlices];
        float M = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kSlices; ++s2) {
          mw[s2] = r0[s2 * PS + HD];
          M = fmaxf(M, mw[s2]);
        }
#pragma unroll
        for (int s2 = 0; s2 < kSlices; ++s2) wgt[s2] = (mw[s2] == -INFINITY) ? 0.0f : exp2f(mw[s2] - M);
        const float Lg = __fadd_rn(__fadd_rn(r0[0 * PS + HD + 1] * wgt[0], r0[1 * PS + HD + 1] * wgt[1]),
                                   __fadd_rn(r0[2 * PS + HD + 1] * wgt[2], r0[3 * PS + HD + 1] * wgt[3]));
        float* pp = a.part + ((static_cast<size_t>(row) * a.H + qh) * a.max_groups + ur.g) * PS;
#pragma unroll
        for (int d2 = 0; d2 < DPL; ++d2) {
          const int d = lane * DPL + d2;
          const float v = __fadd_rn(__fadd_rn(r0[0 * PS + d] * wgt[0], r0[1 * PS + d] * wgt[1]),
                                    __fadd_rn(r0[2 * PS + d] * wgt[2], r0[3 * PS + d] * wgt[3]));
          __stcg(pp + d, v);
        }
        if (lane == 0) {
          __stcg(pp + HD, M);
          __stcg(pp + HD + 1, Lg);
        }
      }
      quad_sync();   // records consumed before the next pass writes them
      buf ^= 1;
    }
    if (sflag[1]) break;
    // the unit that completes an (item, KV head) merges its groups in group order: the
    // barrier orders the team's partial writes before one thread's gpu-scope release
    // increment; the last arriver's acquire makes every unit's partials visible
    team_sync();
    if (tt == 0) {
      int prev;
      asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "l"(a.counters + it.counter * a.KVH + ur.kvh)
                   : "memory");
      sflag[0] = (prev == it.n_groups - 1) ? 1 : 0;
    }
    team_sync();
    if (sflag[0]) {
      for (int qi = cw; qi < nq; qi += kTeamWarps) {
        const int row = it.row_begin + qi / G, qh = ur.kvh * G + qi % G;
        const float* base = a.part + (static_cast<size_t>(row) * a.H + qh) * a.max_groups * PS;
        float mg[2] = {-INFINITY, -INFINITY}, lg[2] = {0.0f, 0.0f};
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int gg = lane + 32 * h2;
          if (gg < it.n_groups) {
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
        for (int d = 0; d < DPL; ++d) O[d] = 0.0f;
        // groups in order; the loads of four groups are issued before their FMAs
        for (int g4 = 0; g4 < it.n_groups; g4 += 4) {
          float pv[4][DPL], wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int gg = g4 + e;
            wv[e] = __shfl_sync(0xffffffffu, gg < 32 ? wg[0] : wg[1], gg & 31);
            if (gg >= it.n_groups) wv[e] = 0.0f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) pv[e][d] = wv[e] != 0.0f ? __ldcg(base + gg * PS + lane * DPL + d) : 0.0f;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (wv[e] == 0.0f) continue;
#pragma unroll
            for (int d = 0; d < DPL; ++d) O[d] = fmaf(wv[e], pv[e][d], O[d]);
          }
        }
        const float invl = 1.0f / Lsum;
        const size_t lo = static_cast<size_t>(a.plane_rows) * a.H * HD;
#pragma unroll
        for (int d = 0; d < DPL; ++d) {
          const size_t o = static_cast<size_t>(row) * a.H * HD + qh * HD + lane * DPL + d;
          store_pair(a.out + o, a.out + lo + o, O[d] * invl);
        }
      }
      if (tt == 0) a.counters[it.counter * a.KVH + ur.kvh] = 0;
    }
  }
  cp_async_wait_all();   // no copy of a skipped pass outlives the CTA
}

template <int HD, int QB>
static cudaError_t launch_attn_variant(cudaLaunchConfig_t cfg, const CUtensorMap& tm, const AttnArgs& a) {
  static bool set = false;
  cfg.dynamicSmemBytes = AttnSmem<HD, QB>::kTotal;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<HD, QB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cfg.dynamicSmemBytes));
    if (e == cudaSuccess) e = apply_carveout(attn_kernel<HD, QB>);
    if (e != cudaSuccess) return e;
    set = true;
  }
  return cudaLaunchKernelEx(&cfg, attn_kernel<HD, QB>, tm, a);
}

template <int HD>
static cudaError_t launch_attn_hd(const cudaLaunchConfig_t& cfg, const CUtensorMap& tm, const AttnArgs& a,
                                  int max_nq) {
  if (max_nq <= 1) return launch_attn_variant<HD, 1>(cfg, tm, a);
  if (max_nq <= 2) return launch_attn_variant<HD, 2>(cfg, tm, a);
  if (max_nq <= 4) return launch_attn_variant<HD, 4>(cfg, tm, a);
  return launch_attn_variant<HD, 8>(cfg, tm, a);
}

size_t attention_smem_bytes(int hd, int max_nq) {
  const int qb = max_nq <= 1 ? 1 : max_nq <= 2 ? 2 : max_nq <= 4 ? 4 : 8;
  if (hd == 128)
    return qb == 1 ? AttnSmem<128, 1>::kTotal : qb == 2 ? AttnSmem<128, 2>::kTotal
                                                          : qb == 4 ? AttnSmem<128, 4>::kTotal : AttnSmem<128, 8>::kTotal;
  return qb == 1 ? AttnSmem<64, 1>::kTotal : qb == 2 ? AttnSmem<64, 2>::kTotal
                                                      : qb == 4 ? AttnSmem<64, 4>::kTotal : AttnSmem<64, 8>::kTotal;
}

cudaError_t launch_attention(const CUtensorMap& tm, const AttnArgs& a, int max_nq, int n_ctas, cudaStream_t st,
                             bool pdl) {
  if (a.n_items <= 0 || a.n_units <= 0) return cudaSuccess;
  if (!a.nodes || !a.items || !a.tails || !a.q || !a.kv_pool || !a.out || !a.part || !a.counters || !a.err ||
      a.plane_rows < 1 || a.max_groups < 1 || a.max_groups > kAttnMaxGroups || max_nq < 1 || n_ctas < 1 ||
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
  if (a.hd == 128) return launch_attn_hd<128>(cfg, tm, a, max_nq);
  return launch_attn_hd<64>(cfg, tm, a, max_nq);
}

}  // namespace dex

// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05) with TMA-fed
// shared-memory pipelines and fused epilogues, for the decoder slices and the shared
// exit head of a DEX round.
//
//   D[row][node] = sum_k W[row][k] * X[node][k]      (W: weights, X: node activations)
//
// Swap-AB: the weights sit on the MMA's M = 128 side, the few lattice nodes of a stage
// batch on the N side (16..256 columns), so each weight byte is read from HBM once per
// round however many nodes the round holds.
//
// Activations arrive as hi/lo bf16 pairs (x ~= hi + lo, two planes of one buffer): each
// 16-wide k step issues W*hi and W*lo into the same fp32 accumulator.  The tensor pipe is
// nearly idle in these weight-streaming GEMMs, so the second MMA costs no time, and the
// activations keep ~17 significant bits instead of bf16's 8.
//
// Persistent, fixed-segment split-K: every 128-row output tile's k range is cut into a
// fixed number of segments S that depends only on the weight shape (and the handle's
// grid), never on the nodes or on how many weight matrices share the launch.  Each
// segment is accumulated from zero; the last CTA to finish one of a tile's segments sums
// them -- fp32 partial tiles in segment order, or (decoder layers of small lattices) the
// exact 2^-32 fixed-point tile sum every segment added at L2 -- and runs the epilogue.  A
// node's result is therefore bit-identical in any batch and in any grouped launch.  The (group, tile, segment) units of a launch are
// dealt out as contiguous ranges over a fixed grid of resident CTAs, so a launch with
// several weight matrices still runs in one wave; each CTA streams its units' k-blocks
// through a deep TMA ring without pausing.  Two TMEM accumulators alternate between
// consecutive units, so the epilogue of one unit overlaps the MMAs of the next.
//
// Roles: warp 0 issues TMA loads (weights first -- they do not depend on the previous
// kernel -- then, after the grid-dependency wait, the activations); warp 1 owns TMEM
// and issues tcgen05.mma; warps 2-5 run the epilogue from TMEM (one accumulator row per
// thread).  Every wait is bounded and reports a stall through the error flag.
//
// Diagnostics: with a.timeline set, epilogue thread 0 of each CTA records its start
// (globaltimer ns, then clock64), the clock64 at which each unit's accumulator was ready
// and at which the unit's epilogue finished, a per-unit tag (bit 0: whole tile, bit 1:
// last arriver that summed the tile, bits 8..15: group, bits 16..31: tile, bits 32..:
// cycles from accumulator-ready to the arrival count), and at the end the clock64 and
// the unit count.
//
// Epilogues: EPI_QKV (RMSNorm scale, RoPE, fp16 K/V into the committed cache or the
// branch pool), EPI_RESID (residual add into the fp32 hidden state, next layer's bf16 input,
// RMSNorm partial sums, exit-head input at a stage boundary), EPI_SWIGLU
// (SiLU(gate) * up), EPI_EXIT (exit logits, DECS mask, Gumbel noise, argmax).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dex {

constexpr int kThreads = 192;
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB weight tile per stage
constexpr int kNtMax = 256;

constexpr int kSumDepth = 2;   // partial tiles whose loads are in flight together in a segment sum

// Split-K segment sums in 2^-32 fixed point: an fp32 partial p with |p| < 2^30 becomes the
// integer nearest p * 2^32 (exact for |p| >= 2^-9, within 2^-33 absolute below), the
// segments' integers add exactly in any order, and the total rounds once to fp32.  A
// partial outside the range (or not finite) adds 0 and raises DEV_RANGE.
constexpr float kFixScale = 4294967296.0f;            // 2^32
constexpr float kFixInv = 2.3283064365386963e-10f;    // 2^-32
constexpr float kFixLimit = 1073741824.0f;            // 2^30
__device__ __forceinline__ long long to_fixed(float p, int32_t* err) {
  if (!(fabsf(p) < kFixLimit)) {
    atomicExch(err, DEV_RANGE);
    return 0;
  }
  return __float2ll_rn(p * kFixScale);
}
__device__ __forceinline__ float from_fixed(long long q) { return __ll2float_rn(q) * kFixInv; }
// fire-and-forget 64-bit add at L2 (two's complement: the unsigned add is the signed one)
__device__ __forceinline__ void red_add_fixed(long long* p, long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(static_cast<unsigned long long>(v))
               : "memory");
}

struct SmemMap {
  size_t a, b, bar, misc, xch, inv, qsum, qkey, total;
};
// Exchange area of the epilogue: 16 accumulator columns x 128 rows (QKV: RoPE partners,
// followed by the group's node table of positions and K/V destinations; SWIGLU: gate/up
// halves; kept for the residual epilogues too, whose launches measured slower with the
// extra ring stage a smaller area allows), a small node table for the exit head (which
// gains a third ring stage at 64-node tiles).
struct QkvNode {
  long long base;   // element offset of the node's (K, head 0, dim 0) entry in its cache
  int pos;          // input position (RoPE row)
  int commit;       // 1: committed cache, 0: branch pool
};
static_assert(sizeof(QkvNode) == 16, "16-byte node table entries");
__host__ __device__ constexpr size_t xch_bytes(int epi) {
  return epi == EPI_EXIT ? 512
                         : static_cast<size_t>(16) * kBM * 4 + (epi == EPI_QKV ? kNtMax * sizeof(QkvNode) : 0);
}
__host__ __device__ inline SmemMap smem_map(int nt, int stages, int epi) {
  SmemMap m;
  m.a = 0;
  m.b = m.a + static_cast<size_t>(stages) * kABytes;
  m.bar = m.b + static_cast<size_t>(stages) * 2 * nt * kBK * 2;   // hi and lo boxes per stage
  m.misc = m.bar + static_cast<size_t>(2 * stages + 4) * 8;       // full, empty, accf[2], tfree[2]
  m.xch = (m.misc + 32 + 15) & ~static_cast<size_t>(15);        // tmem slot + flags
  m.inv = m.xch + xch_bytes(epi);
  m.qsum = m.inv + kNtMax * 4;
  m.qkey = m.qsum + 4 * 16 * 4;
  m.total = m.qkey + 4 * 16 * 8;
  return m;
}

size_t gemm_smem_bytes(int nt, int stages, int epi) { return smem_map(nt, stages, epi).total + 1024; }

constexpr size_t kSmemOptin = 227 * 1024;   // largest dynamic shared memory a CTA may opt into

// Pipeline depth: the most stages (2..8) whose whole footprint fits the given budget for
// small node tiles, or the opt-in limit for the wide tiles of prefill.
int gemm_stages_for(int nt, int epi, size_t small_budget) {
  const size_t budget = nt <= 64 ? small_budget : kSmemOptin;
  int s = 8;
  while (s > 2 && gemm_smem_bytes(nt, s, epi) > budget) --s;
  return s;
}

// Units of a launch, group-major: u = (g * n_tiles + t) * S + s.  CTA c owns units
// [c U / C, (c+1) U / C).  Segment s of a tile covers k-blocks [s kb / S, (s+1) kb / S).
struct Unit {
  int g, t, s, k0, k1;
};
__device__ __forceinline__ Unit unit_at(int u, int n_tiles, int S, int kb) {
  Unit x;
  const int per_group = n_tiles * S;
  x.g = u / per_group;
  const int r = u - x.g * per_group;
  x.t = r / S;
  x.s = r - x.t * S;
  x.k0 = (x.s * kb) / S;
  x.k1 = ((x.s + 1) * kb) / S;
  return x;
}
__device__ __forceinline__ int unit_begin(int c, int U, int C) {
  return static_cast<int>((static_cast<long long>(c) * U) / C);
}

// Segments per tile for a weight shape on a grid of C CTAs: the smallest S for which the
// busiest CTA of a one-matrix launch streams at most 1/0.9 of the average k-blocks (fewer
// segments mean fewer partial tiles to write and sum), else the best balance among
// S <= 8 C / n_tiles.  Host-side, once per handle.
int gemm_segments(int n_tiles, int kblocks, int C) {
  int best = 1;
  double best_eff = -1.0;
  const int s_max = std::max(1, std::min(kblocks, (8 * C + n_tiles - 1) / n_tiles));
  const double avg = static_cast<double>(n_tiles) * kblocks / C;
  for (int S = 1; S <= s_max; ++S) {
    const long long U = static_cast<long long>(n_tiles) * S;
    long long most = 0;
    for (int c = 0; c < C; ++c) {
      const long long u0 = c * U / C, u1 = (c + 1) * U / C;
      long long w = 0;
      for (long long u = u0; u < u1; ++u) {
        const long long sg = u % S;
        w += ((sg + 1) * kblocks) / S - (sg * kblocks) / S;
      }
      most = std::max(most, w);
    }
    const double eff = most > 0 ? avg / static_cast<double>(most) : 0.0;
    if (eff >= 0.9) return S;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = S;
    }
  }
  return best;
}

// Two CTAs per SM must stay resident (the persistent grid is 2 x SMs): at most 170
// registers per thread.
// Epilogues that may take their k segments' sum from the fixed-point tile sums (the
// decoder layers); the exit head and the adapters always sum fp32 partials.
template <int EPI>
__host__ __device__ constexpr bool red_sum_epi() {
  return EPI == EPI_QKV || EPI == EPI_RESID || EPI == EPI_SWIGLU;
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ GemmArgs a) {
  constexpr bool kRedOk = red_sum_epi<EPI>();
  const int C = gridDim.x, cta = blockIdx.x;
  const int kb = a.kblocks, S = a.n_segs, nT = a.n_tiles;
  const int U = a.n_groups * nT * S;
  const int u0 = unit_begin(cta, U, C), u1 = unit_begin(cta + 1, U, C);
  if (u0 >= u1) return;   // no work (more CTAs than units)
  const int n_units = u1 - u0;
  int nwork = 0;   // k-blocks this CTA streams
  for (int u = u0; u < u1; ++u) {
    const Unit x = unit_at(u, nT, S, kb);
    nwork += x.k1 - x.k0;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemMap sm = smem_map(a.nt, a.stages, EPI);
  uint8_t* sA = smem + sm.a;
  uint8_t* sB = smem + sm.b;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + sm.bar);
  uint64_t* empty = full + a.stages;
  uint64_t* accf = empty + a.stages;   // [2] accumulator ready
  uint64_t* tfree = accf + 2;          // [2] accumulator drained by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + sm.misc);
  volatile int* sflag = reinterpret_cast<volatile int*>(smem + sm.misc + 4);   // [0] last, [1] abort
  float* xch = reinterpret_cast<float*>(smem + sm.xch);
  float* inv = reinterpret_cast<float*>(smem + sm.inv);
  float* qsum = reinterpret_cast<float*>(smem + sm.qsum);
  unsigned long long* qkey = reinterpret_cast<unsigned long long*>(smem + sm.qkey);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int stages = a.stages;
  const uint32_t b_bytes = static_cast<uint32_t>(a.nt) * kBK * 2;
  const uint32_t cols = static_cast<uint32_t>(a.tmem_cols);

  auto tile_src = [&](int t, int& src, int& lt) {
    src = 0;
    lt = t;
    if (t >= a.src_tiles0 + a.src_tiles1) {
      src = 2;
      lt = t - a.src_tiles0 - a.src_tiles1;
    } else if (t >= a.src_tiles0) {
      src = 1;
      lt = t - a.src_tiles0;
    }
  };

  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&tfree[b], 128);
    }
    sflag[0] = 0;
    sflag[1] = 0;
    fence_mbar_init();
    if (!a.groups[0].a_packed) {
      tma_prefetch(&tmA0);
      if (a.src_tiles0 < a.n_tiles || EPI == EPI_SWIGLU) tma_prefetch(&tmA1);
      if (a.src_tiles0 + a.src_tiles1 < a.n_tiles) tma_prefetch(&tmA2);
    }
    tma_prefetch(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      auto load_a = [&](const Unit& x, int k, int st) {
        uint8_t* dst = sA + static_cast<size_t>(st) * kABytes;
        const uint8_t* packed = a.groups[x.g].a_packed;
        if (packed) {   // packed weights: the (tile, k-block) 16 KB box is contiguous
          const uint8_t* src = packed + (static_cast<size_t>(x.t) * kb + k) * kABytes;
          if (a.evict_first) bulk_load_1d_hint(dst, src, kABytes, &full[st], pol);
          else bulk_load_1d(dst, src, kABytes, &full[st]);
          return;
        }
        const int kx = k * kBK;
        int src, lt;
        tile_src(x.t, src, lt);
        if (EPI == EPI_SWIGLU) {
          if (a.evict_first) {
            tma_load_2d_hint(dst, &tmA0, &full[st], kx, lt * 64, pol);
            tma_load_2d_hint(dst + kABytes / 2, &tmA1, &full[st], kx, lt * 64, pol);
          } else {
            tma_load_2d(dst, &tmA0, &full[st], kx, lt * 64);
            tma_load_2d(dst + kABytes / 2, &tmA1, &full[st], kx, lt * 64);
          }
        } else {
          const CUtensorMap* mapA = src == 0 ? &tmA0 : (src == 1 ? &tmA1 : &tmA2);
          if (a.evict_first) tma_load_2d_hint(dst, mapA, &full[st], kx, lt * kBM, pol);
          else tma_load_2d(dst, mapA, &full[st], kx, lt * kBM);
        }
      };
      auto load_b = [&](const Unit& x, int k, int st) {   // hi box, then the lo box plane_rows rows further
        uint8_t* dst = sB + static_cast<size_t>(st) * 2 * b_bytes;
        const int row0 = a.groups[x.g].b_row0;
        tma_load_2d(dst, &tmB, &full[st], k * kBK, row0);
        tma_load_2d(dst + b_bytes, &tmB, &full[st], k * kBK, row0 + a.plane_rows);
      };
      // weights of the first ring slots before the grid-dependency wait
      const int npre = nwork < stages ? nwork : stages;
      {
        int u = u0, i = 0;
        Unit x = unit_at(u, nT, S, kb);
        int k = x.k0;
        for (; i < npre; ++i) {
          mbar_arrive_expect_tx(&full[i], kABytes + 2 * b_bytes);
          load_a(x, k, i);
          if (++k == x.k1 && ++u < u1) {
            x = unit_at(u, nT, S, kb);
            k = x.k0;
          }
        }
      }
      griddep_wait();   // activations are produced by the previous kernel
      int u = u0;
      Unit x = unit_at(u, nT, S, kb);
      int k = x.k0;
      int issued = npre;
      bool ok = true;
      for (int i = 0; i < nwork; ++i) {
        const int st = i % stages;
        if (i >= npre) {
          const uint32_t use = static_cast<uint32_t>(i / stages);
          if (!mbar_wait(&empty[st], (use - 1) & 1u, a.err, DEV_TIMEOUT_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], kABytes + 2 * b_bytes);
          load_a(x, k, st);
          issued = i + 1;
        }
        load_b(x, k, st);
        if (++k == x.k1 && ++u < u1) {
          x = unit_at(u, nT, S, kb);
          k = x.k0;
        }
      }
      if (!ok) {   // drain copies still in flight before the CTA can exit
        for (int i = (issued > stages ? issued - stages : 0); i < issued; ++i)
          mbar_wait(&full[i % stages], static_cast<uint32_t>(i / stages) & 1u, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, a.nt);
      int ui = 0;   // unit index within this CTA
      int u = u0;
      Unit x = unit_at(u, nT, S, kb);
      int k = x.k0;
      for (int i = 0; i < nwork; ++i) {
        const bool seg_first = (k == x.k0);
        const bool seg_last = (k == x.k1 - 1);
        const int buf = ui & 1;
        if (seg_first && ui >= 2) {   // reuse of an accumulator: wait until the epilogue drained it
          if (!mbar_wait(&tfree[buf], static_cast<uint32_t>((ui >> 1) - 1) & 1u, a.err, DEV_TIMEOUT_ACC)) break;
          tc_fence_after();
        }
        const int st = i % stages;
        if (!mbar_wait(&full[st], static_cast<uint32_t>(i / stages) & 1u, a.err, DEV_TIMEOUT_FULL)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf) * cols;
        const uint32_t abase = smem_u32(sA + static_cast<size_t>(st) * kABytes);
        const uint32_t bbase = smem_u32(sB + static_cast<size_t>(st) * 2 * b_bytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t adesc = sw128_kmajor_desc(abase + kk * 32);
          umma_bf16(d, adesc, sw128_kmajor_desc(bbase + kk * 32), idesc, (!seg_first || kk > 0) ? 1u : 0u);
          umma_bf16(d, adesc, sw128_kmajor_desc(bbase + b_bytes + kk * 32), idesc, 1u);
        }
        umma_commit(&empty[st]);
        if (seg_last) {
          umma_commit(&accf[buf]);
          ++ui;
        }
        if (++k == x.k1 && ++u < u1) {
          x = unit_at(u, nT, S, kb);
          k = x.k0;
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int wq = warp & 3;           // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;      // accumulator row within the tile
    const int ep = tid - 64;           // 0..127
    const int ndt = a.d / 128;
    unsigned long long* tl = (a.timeline && ep == 0) ? a.timeline + static_cast<size_t>(cta) * kTimelineSlots : nullptr;
    if (tl) {
      tl[0] = global_timer_ns();
      tl[1] = clock64();
    }
    griddep_wait();
    int g_inv = -1;                    // group whose RMSNorm scales are in inv[]

    // per-chunk epilogue of tile (src, lt) of group g: v[j] = accumulator of (row r, node c0 + j)
    auto epilogue_chunk = [&](const GemmGroup& grp, int src, int lt, int c0, float (&v)[16]) {
      const int n = grp.n;
      const int b_row0 = grp.b_row0;
      if (EPI == EPI_QKV) {
        const int f = lt * kBM + r;      // feature within the source (q, k or v)
        const int half = a.hd >> 1;
        const QkvNode* ntab = reinterpret_cast<const QkvNode*>(xch + 16 * kBM);
#pragma unroll
        for (int j = 0; j < 16; ++j) xch[j * kBM + r] = (c0 + j < n) ? v[j] * inv[c0 + j] : 0.0f;
        named_bar_sync(1, 128);
        const int head = f / a.hd, dim = f - head * a.hd;
        // the chunk's RoPE factors, all loads issued before the arithmetic
        float2 cs[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          cs[j] = make_float2(1.0f, 0.0f);
          if (src != 2 && c0 + j < n)
            cs[j] = __ldg(a.rope + static_cast<size_t>(ntab[c0 + j].pos) * half + (dim & (half - 1)));
        }
        const int kv = src - 1;
        const size_t off_commit = static_cast<size_t>(kv * a.KVH + head) * a.max_ctx * a.hd + dim;
        const size_t off_pool = static_cast<size_t>(kv * a.KVH + head) * a.hd + dim;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + j;
          if (c < n) {
            const float x = xch[j * kBM + r];
            float out = x;
            if (src != 2) {
              const float y = xch[j * kBM + (r ^ half)];
              out = dim < half ? x * cs[j].x - y * cs[j].y : x * cs[j].x + y * cs[j].y;
            }
            if (src == 0) {
              a.q_out[static_cast<size_t>(b_row0 + c) * (a.H * a.hd) + f] = out;
            } else {
              const QkvNode nd = ntab[c];
              __half* dst = nd.commit ? a.kv_commit + nd.base + off_commit : a.kv_pool + nd.base + off_pool;
              *dst = __float2half_rn(out);   // the caches hold fp16 K/V
            }
          }
        }
        named_bar_sync(1, 128);
      } else if (EPI == EPI_RESID) {
        const int f = lt * kBM + r;
        const int* hrow = reinterpret_cast<const int*>(inv);
        // every load of the chunk first: hidden state of the 16 nodes, the two gains
        float hv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          hv[j] = (c0 + j < n) ? a.hidden[static_cast<size_t>(hrow[c0 + j]) * a.d + f] : 0.0f;
        const float gn = grp.has_next ? bf16_to_f32(grp.g_next[f]) : 0.0f;
        const float ge = grp.stage_end ? bf16_to_f32((grp.g_exit ? grp.g_exit : a.g_final)[f]) : 0.0f;
        float sq[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + j;
          sq[j] = 0.0f;
          if (c < n) {
            const float x = __fadd_rn(hv[j], v[j]);
            a.hidden[static_cast<size_t>(hrow[c]) * a.d + f] = x;
            const size_t o = static_cast<size_t>(b_row0 + c) * a.d + f;
            const size_t lo = static_cast<size_t>(a.plane_rows) * a.d;
            if (grp.has_next) store_pair(a.hb_out + o, a.hb_out + lo + o, __fmul_rn(x, gn));
            if (grp.stage_end) store_pair(a.exit_hb + o, a.exit_hb + lo + o, __fmul_rn(x, ge));
            sq[j] = __fmul_rn(x, x);
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float s = warp_sum(sq[j]);
          if (lane == 0) qsum[wq * 16 + j] = s;
        }
        named_bar_sync(1, 128);
        if (ep < 16 && c0 + ep < n) {
          const float t = __fadd_rn(__fadd_rn(qsum[0 * 16 + ep], qsum[1 * 16 + ep]),
                                    __fadd_rn(qsum[2 * 16 + ep], qsum[3 * 16 + ep]));
          const size_t o = static_cast<size_t>(b_row0 + c0 + ep) * ndt + lt;
          a.ssq_out[o] = t;
          if (grp.stage_end) a.exit_ssq[o] = t;
        }
        named_bar_sync(1, 128);
      } else if (EPI == EPI_SWIGLU) {
#pragma unroll
        for (int j = 0; j < 16; ++j) xch[j * kBM + r] = (c0 + j < n) ? v[j] * inv[c0 + j] : 0.0f;
        named_bar_sync(1, 128);
        const int feat = lt * 64 + (r & 63);
        if (r < 64 && feat < a.d_ff) {
          for (int j = 0; j < 16; ++j) {
            const int c = c0 + j;
            if (c >= n) break;
            const float g = xch[j * kBM + r], u = xch[j * kBM + r + 64];
            const float act = g / (1.0f + expf(-g)) * u;
            const size_t o = static_cast<size_t>(b_row0 + c) * a.d_ff + feat;
            store_pair(a.act_out + o, a.act_out + static_cast<size_t>(a.plane_rows) * a.d_ff + o, act);
          }
        }
        named_bar_sync(1, 128);
      } else if (EPI == EPI_ADUP) {   // adapter layer 1: SiLU(W1 RMSNorm(h; g) + b1)
        const int f = lt * kBM + r;      // hidden unit of the adapter (0 .. 2d-1)
        const float b1 = bf16_to_f32(grp.bias[f]);
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + j;
          if (c >= n) break;
          const float u = __fadd_rn(v[j] * inv[c], b1);
          const float act = u / (1.0f + expf(-u));
          const size_t o = static_cast<size_t>(b_row0 + c) * a.d_ff + f;
          store_pair(a.act_out + o, a.act_out + static_cast<size_t>(a.plane_rows) * a.d_ff + o, act);
        }
      } else if (EPI == EPI_ADDOWN) {   // adapter layer 2: h~ = h + alpha (W2 a + b2) -> exit input
        const int f = lt * kBM + r;
        const float b2 = bf16_to_f32(grp.bias[f]);
        const float gf = bf16_to_f32(a.g_final[f]);
        float sq[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + j;
          sq[j] = 0.0f;
          if (c < n) {
            const float x = __fadd_rn(a.hidden[static_cast<size_t>(reinterpret_cast<const int*>(inv)[c]) * a.d + f],
                                      __fmul_rn(grp.alpha, __fadd_rn(v[j], b2)));
            const size_t o = static_cast<size_t>(b_row0 + c) * a.d + f;
            store_pair(a.exit_hb + o, a.exit_hb + static_cast<size_t>(a.plane_rows) * a.d + o, __fmul_rn(x, gf));
            sq[j] = __fmul_rn(x, x);
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float s = warp_sum(sq[j]);
          if (lane == 0) qsum[wq * 16 + j] = s;
        }
        named_bar_sync(1, 128);
        if (ep < 16 && c0 + ep < n)
          a.exit_ssq[static_cast<size_t>(b_row0 + c0 + ep) * ndt + lt] =
              __fadd_rn(__fadd_rn(qsum[0 * 16 + ep], qsum[1 * 16 + ep]), __fadd_rn(qsum[2 * 16 + ep], qsum[3 * 16 + ep]));
        named_bar_sync(1, 128);
      } else {   // EPI_EXIT
        // The chunk's 16 nodes: sequence, target position and the DECS mask restricted to this
        // tile's 128 vocabulary rows (a bitmap), staged in shared memory by 16 threads.
        int* cm = reinterpret_cast<int*>(xch);   // [0,16) seq, [16,32) target pos, [32,96) mask words
        if (ep < 16) {
          const int c = c0 + ep;
          uint32_t mw[4] = {0u, 0u, 0u, 0u};
          int seq = 0, tpos = 0;
          if (c < n) {
            const DevNode* nd = a.nodes + b_row0 + c;
            seq = nd->seq;
            tpos = nd->target_pos;
            if (!nd->unmasked) {
              for (int p = 0; p < nd->n_prior; ++p) {
                const int t = a.priors[nd->prior_off + p] - lt * kBM;
                if (t >= 0 && t < kBM) mw[t >> 5] |= 1u << (t & 31);
              }
            }
          }
          cm[ep] = seq;
          cm[16 + ep] = tpos;
#pragma unroll
          for (int k = 0; k < 4; ++k) cm[32 + 4 * ep + k] = static_cast<int>(mw[k]);
        }
        named_bar_sync(1, 128);
        const uint32_t vid = static_cast<uint32_t>(lt * kBM + r);
        const bool v_ok = vid < static_cast<uint32_t>(a.vocab);
        float noise[16];
        if (a.sample) {
          // Gumbel rows: one Philox4x32-10 block covers four consecutive vocabulary entries, so
          // lane 4k+m computes the block of node 4g+m for its quad's entries, and a 4x4 transpose
          // within the quad gives every lane its own entry's word for the four nodes
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int jn = 4 * g + (lane & 3);
            const U4 w4 = philox4x32_10(U4{vid >> 2, static_cast<uint32_t>(cm[16 + jn]), static_cast<uint32_t>(cm[jn]),
                                           0x44455843u},
                                        static_cast<uint32_t>(a.seed), static_cast<uint32_t>(a.seed >> 32));
            const bool b1 = lane & 2, b0 = lane & 1;
            // round 1 (lanes m, m^2): keep the half of the row the lane's column pair needs
            const uint32_t r0 = __shfl_xor_sync(0xffffffffu, b1 ? w4.x : w4.z, 2);
            const uint32_t r1 = __shfl_xor_sync(0xffffffffu, b1 ? w4.y : w4.w, 2);
            const uint32_t B0 = b1 ? r0 : w4.x, B1 = b1 ? r1 : w4.y, B2 = b1 ? w4.z : r0, B3 = b1 ? w4.w : r1;
            // round 2 (lanes m, m^1)
            const uint32_t t0 = __shfl_xor_sync(0xffffffffu, b0 ? B0 : B1, 1);
            const uint32_t t1 = __shfl_xor_sync(0xffffffffu, b0 ? B2 : B3, 1);
            const uint32_t C[4] = {b0 ? t0 : B0, b0 ? B1 : t0, b0 ? t1 : B2, b0 ? B3 : t1};
#pragma unroll
            for (int e = 0; e < 4; ++e) noise[4 * g + e] = gumbel_from_bits(C[e]);
          }
        }
        unsigned long long key[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + j;
          float score = -INFINITY;
          if (c < n && v_ok) {
            const float logit = v[j] * inv[c];
            if (a.logits_dbg) a.logits_dbg[static_cast<size_t>(b_row0 + c) * a.vocab + vid] = logit;
            const bool masked = (static_cast<uint32_t>(cm[32 + 4 * j + (r >> 5)]) >> (r & 31)) & 1u;
            if (!masked) score = a.sample ? logit / a.tau + noise[j] : logit;
          }
          key[j] = argmax_key(score, vid);
        }
        const unsigned long long best_key = warp_argmax16_transposed(key, lane);   // node lane / 2
        if ((lane & 1) == 0) qkey[wq * 16 + (lane >> 1)] = best_key;
        named_bar_sync(1, 128);
        if (ep < 16 && c0 + ep < n) {
          unsigned long long k = qkey[ep];
          for (int w = 1; w < 4; ++w) k = qkey[w * 16 + ep] > k ? qkey[w * 16 + ep] : k;
          atomicMax(a.best + b_row0 + c0 + ep, k);
        }
        named_bar_sync(1, 128);
      }
    };

    for (int ui = 0; ui < n_units; ++ui) {
      const Unit x = unit_at(u0 + ui, nT, S, kb);
      const GemmGroup& grp = a.groups[x.g];
      const int n = grp.n;
      const int buf = ui & 1;
      int src, lt;
      tile_src(x.t, src, lt);
      if ((EPI == EPI_RESID || EPI == EPI_ADDOWN) && x.g != g_inv) {   // hidden-state rows of the group's nodes
        named_bar_sync(1, 128);                 // previous readers of the table are done
        for (int c = ep; c < n; c += 128) reinterpret_cast<int*>(inv)[c] = a.nodes[grp.b_row0 + c].hrow;
        g_inv = x.g;
      }
      if (EPI != EPI_RESID && EPI != EPI_ADDOWN && x.g != g_inv) {   // RMSNorm scales of this group's node rows
        named_bar_sync(1, 128);                 // previous readers of inv[] are done
        for (int c = ep; c < n; c += 128) {
          const float* sp = a.ssq_in + static_cast<size_t>(grp.b_row0 + c) * ndt;
          float t = sp[0];
          for (int j = 1; j < ndt; ++j) t = __fadd_rn(t, sp[j]);
          inv[c] = 1.0f / sqrtf(__fadd_rn(__fdiv_rn(t, static_cast<float>(a.d)), a.eps));
          if (EPI == EPI_QKV) {   // where the node's K and V go, and its RoPE row
            const DevNode* nd = a.nodes + grp.b_row0 + c;
            QkvNode e;
            e.pos = nd->pos;
            e.commit = nd->kv_commit;
            e.base = e.commit
                         ? static_cast<long long>(((static_cast<size_t>(nd->seq) * a.L + grp.layer) * 2 * a.KVH) *
                                                      a.max_ctx + e.pos) * a.hd
                         : static_cast<long long>(((static_cast<size_t>(nd->seq) * a.n_slots + nd->slot) * a.L +
                                                   grp.layer) * 2 * a.KVH) * a.hd;
            reinterpret_cast<QkvNode*>(xch + 16 * kBM)[c] = e;
          }
        }
        g_inv = x.g;
      }
      if (!mbar_wait(&accf[buf], static_cast<uint32_t>(ui >> 1) & 1u, a.err, DEV_TIMEOUT_ACC)) sflag[1] = 1;
      const bool rec = tl && ui < kTimelineUnits;
      if (rec) tl[4 + 3 * ui] = clock64();
      named_bar_sync(1, 128);
      if (sflag[1]) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(buf) * cols + (static_cast<uint32_t>(wq * 32) << 16);
      if (S == 1) {   // the whole tile is this unit
        for (int c0 = 0; c0 < n; c0 += 16) {
          float v[16];
          tmem_ld16(taddr + static_cast<uint32_t>(c0), v);
          epilogue_chunk(grp, src, lt, c0, v);
        }
        tc_fence_before();
        mbar_arrive(&tfree[buf]);
        if (rec) {
          tl[5 + 3 * ui] = clock64();
          tl[6 + 3 * ui] = 1ull | (static_cast<unsigned long long>(x.g) << 8) |
                           (static_cast<unsigned long long>(x.t & 0xffff) << 16);
        }
      } else {
        const size_t tile_id = static_cast<size_t>(x.g) * nT + x.t;
        // tile sums (red path): column c of this thread's row at acc_row[c * kBM]
        long long* acc_row = (kRedOk && a.sum_mode == SUM_FIXED_RED) ? a.acc + tile_id * a.nt * kBM + r : nullptr;
        // segment partials: [unit][row][nt] fp32, a thread's 16 columns are 64 contiguous bytes
        const size_t tile_unit0 = tile_id * S;   // unit of segment 0
        for (int c0 = 0; c0 < n; c0 += 16) {
          float v[16];
          tmem_ld16(taddr + static_cast<uint32_t>(c0), v);
          if (kRedOk && acc_row) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < n) red_add_fixed(acc_row + static_cast<size_t>(c0 + j) * kBM, to_fixed(v[j], a.err));
            if (EPI == EPI_RESID) {   // the residual rows the last arriver reads, while the arrival runs
              const int* hrow = reinterpret_cast<const int*>(inv);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < n) prefetch_l1(a.hidden + static_cast<size_t>(hrow[c0 + j]) * a.d + lt * kBM + r);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(a.partial + ((tile_unit0 + x.s) * kBM + r) * a.nt + c0);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              __stcg(dst + q4, make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]));
          }
        }
        tc_fence_before();
        mbar_arrive(&tfree[buf]);
        // arrival: the CTA barrier orders every thread's partial (or red) before one thread's
        // gpu-scope acq_rel increment, which releases them to the last arriver and, for the
        // last arriver, acquires the other segments' (the second barrier passes that on)
        named_bar_sync(1, 128);
        int32_t* counter = a.counters + tile_id;
        if (ep == 0) {
          int prev;
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(counter) : "memory");
          sflag[0] = (prev == S - 1) ? 1 : 0;
        }
        named_bar_sync(1, 128);
        const unsigned long long t_arrived = rec ? clock64() : 0ull;
        if (!acc_row && sflag[0]) {   // last of the tile's segments: fp32 partials in segment order
          // (the exit head's epilogue leaves registers for one partial tile in flight)
          constexpr int kDepth = EPI == EPI_EXIT ? 1 : kSumDepth;
          const size_t seg_f4 = static_cast<size_t>(kBM) * a.nt / 4;
          const float4* prow = reinterpret_cast<const float4*>(a.partial + (tile_unit0 * kBM + r) * a.nt);
          for (int c0 = 0; c0 < n; c0 += 16) {
            float v[16];
            const float4* pc = prow + c0 / 4;
            for (int s0 = 0; s0 < S; s0 += kDepth) {
              float4 q[kDepth][4];
#pragma unroll
              for (int i = 0; i < kDepth; ++i)
                if (s0 + i < S) {
#pragma unroll
                  for (int q4 = 0; q4 < 4; ++q4) q[i][q4] = __ldcg(pc + (s0 + i) * seg_f4 + q4);
                }
#pragma unroll
              for (int i = 0; i < kDepth; ++i)
                if (s0 + i < S) {
                  const bool first = (s0 + i == 0);
#pragma unroll
                  for (int q4 = 0; q4 < 4; ++q4) {
                    v[4 * q4 + 0] = first ? q[i][q4].x : __fadd_rn(v[4 * q4 + 0], q[i][q4].x);
                    v[4 * q4 + 1] = first ? q[i][q4].y : __fadd_rn(v[4 * q4 + 1], q[i][q4].y);
                    v[4 * q4 + 2] = first ? q[i][q4].z : __fadd_rn(v[4 * q4 + 2], q[i][q4].z);
                    v[4 * q4 + 3] = first ? q[i][q4].w : __fadd_rn(v[4 * q4 + 3], q[i][q4].w);
                  }
                }
            }
            epilogue_chunk(grp, src, lt, c0, v);
          }
          if (ep == 0) *counter = 0;
        } else if (kRedOk && sflag[0]) {   // last of the tile's segments: the exact fixed-point sum, then the epilogue
          for (int c0 = 0; c0 < n; c0 += 16) {
            long long t64[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              t64[j] = (c0 + j < n) ? __ldcg(acc_row + static_cast<size_t>(c0 + j) * kBM) : 0ll;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < n) __stcg(acc_row + static_cast<size_t>(c0 + j) * kBM, 0ll);   // zero at rest
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = from_fixed(t64[j]);
            epilogue_chunk(grp, src, lt, c0, v);
          }
          if (ep == 0) *counter = 0;
        }
        named_bar_sync(1, 128);
        if (rec) {
          tl[5 + 3 * ui] = clock64();
          tl[6 + 3 * ui] = (sflag[0] ? 2ull : 0ull) | (static_cast<unsigned long long>(x.g) << 8) |
                           (static_cast<unsigned long long>(x.t & 0xffff) << 16) |
                           ((t_arrived - tl[4 + 3 * ui]) << 32);
        }
      }
    }
    if (tl) {
      tl[2] = clock64();
      tl[3] = static_cast<unsigned long long>(n_units);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * cols);
  }
}

template <int EPI>
static cudaError_t launch_one(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& a2,
                              const CUtensorMap& b, const GemmArgs& args, cudaStream_t st, bool pdl) {
  static bool attr_set = false;
  const size_t smem = gemm_smem_bytes(args.nt, args.stages, EPI);
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemOptin));
    if (e == cudaSuccess) e = apply_carveout(gemm_tc_kernel<EPI>);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(args.n_ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<EPI>, a0, a1, a2, b, args);
}

cudaError_t launch_gemm(int epi, const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& a2,
                        const CUtensorMap& b, const GemmArgs& args, cudaStream_t st, bool pdl) {
  if (args.nt < 16 || args.nt > kNtMax || (args.nt & 15) || args.n_groups < 1 || args.n_groups > kMaxGroups ||
      args.n_ctas < 1 || args.n_segs < 1 || args.n_segs > args.kblocks || args.n_tiles < 1 || args.kblocks < 1 ||
      static_cast<long long>(args.n_groups) * args.n_tiles * args.n_segs > (1ll << 30))
    return cudaErrorInvalidValue;
  // a launch mixes packed groups with tensor-map weights never: the prefetch decision is per launch
  for (int g = 1; g < args.n_groups; ++g)
    if ((args.groups[g].a_packed != nullptr) != (args.groups[0].a_packed != nullptr)) return cudaErrorInvalidValue;
  // every pointer the chosen epilogue dereferences must be set (checked here, on the host)
  bool any_next = false, any_end = false;
  for (int g = 0; g < args.n_groups; ++g) {
    const GemmGroup& gr = args.groups[g];
    if (gr.n < 1 || gr.n > args.nt || gr.b_row0 < 0 || gr.b_row0 + gr.n > args.plane_rows)
      return cudaErrorInvalidValue;
    if (gr.has_next && !gr.g_next) return cudaErrorInvalidValue;
    any_next |= gr.has_next != 0;
    any_end |= gr.stage_end != 0;
  }
  if (!args.err || !args.counters || !args.partial) return cudaErrorInvalidValue;
  const bool red_ok = epi == EPI_QKV || epi == EPI_RESID || epi == EPI_SWIGLU;
  if (args.sum_mode != SUM_FP32 && (args.sum_mode != SUM_FIXED_RED || !red_ok || !args.acc))
    return cudaErrorInvalidValue;
  if (epi != EPI_RESID && epi != EPI_ADDOWN && !args.ssq_in) return cudaErrorInvalidValue;
  if (epi != EPI_SWIGLU && epi != EPI_ADUP && !args.nodes) return cudaErrorInvalidValue;
  if (epi == EPI_ADUP || epi == EPI_ADDOWN)
    for (int g = 0; g < args.n_groups; ++g)
      if (!args.groups[g].bias) return cudaErrorInvalidValue;
  if (epi == EPI_ADUP && !args.act_out) return cudaErrorInvalidValue;
  if (epi == EPI_ADDOWN && (!args.hidden || !args.exit_hb || !args.exit_ssq || !args.g_final))
    return cudaErrorInvalidValue;
  if (epi == EPI_QKV && (!args.q_out || !args.kv_commit || !args.kv_pool || !args.rope)) return cudaErrorInvalidValue;
  if (epi == EPI_RESID && (!args.hidden || !args.ssq_out || (any_next && !args.hb_out) ||
                           (any_end && (!args.exit_hb || !args.exit_ssq || !args.g_final))))
    return cudaErrorInvalidValue;
  if (epi == EPI_SWIGLU && !args.act_out) return cudaErrorInvalidValue;
  if (epi == EPI_EXIT && !args.best) return cudaErrorInvalidValue;
  if (args.tmem_cols < args.nt || args.tmem_cols < 32 || args.tmem_cols > 256 ||
      (args.tmem_cols & (args.tmem_cols - 1)))
    return cudaErrorInvalidValue;
  if (args.stages < 2 || args.stages > 8 || gemm_smem_bytes(args.nt, args.stages, epi) > kSmemOptin)
    return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_QKV: return launch_one<EPI_QKV>(a0, a1, a2, b, args, st, pdl);
    case EPI_RESID: return launch_one<EPI_RESID>(a0, a1, a2, b, args, st, pdl);
    case EPI_SWIGLU: return launch_one<EPI_SWIGLU>(a0, a1, a2, b, args, st, pdl);
    case EPI_EXIT: return launch_one<EPI_EXIT>(a0, a1, a2, b, args, st, pdl);
    case EPI_ADUP: return launch_one<EPI_ADUP>(a0, a1, a2, b, args, st, pdl);
    case EPI_ADDOWN: return launch_one<EPI_ADDOWN>(a0, a1, a2, b, args, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dex

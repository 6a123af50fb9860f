// C ABI of the DEX library (include/dex.h): handle life cycle, prefill, DEX / AR rounds,
// statistics, and the isolated exit-head and collapse entry points.
//
// A round ("Depth Exploration for LLM Decoding", Algorithm 1, one loop iteration):
//   plan (host lattice FSM) -> upload node tables -> pending collapse copies ->
//   stage-input assembly -> for each live stage s, layers (d_{s-1}, d_s] over the stage's
//   nodes (QKV + RoPE + KV write, lattice attention, O + residual, gate/up + SwiGLU,
//   down + residual) -> exit head + DECS over every node -> one device-to-host read of
//   the tokens -> insert / validate_and_commit / collapse on the host.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <map>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/dex.h"
#include "common.cuh"
#include "kernels.h"
#include "lattice.h"

using bf16 = __nv_bfloat16;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder() {
  if (g_encode) return DEX_OK;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return DEX_ECUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return DEX_OK;
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix, box {64 cols, box_rows},
// 128-byte swizzle, zero fill out of bounds.
int encode_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (cols * 2) % 16) return DEX_EINVAL;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DEX_OK : DEX_EINVAL;
}

int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

constexpr int kPrefillRowsMax = 512;   // most prompt positions per prefill pass (rows of the scratch planes)

struct dex_handle {
  // model
  int L = 0, d = 0, H = 0, KVH = 0, hd = 0, dff = 0, V = 0;
  float eps = 0, theta = 0;
  const bf16* embed = nullptr;
  const bf16* final_norm = nullptr;
  const bf16* lm_head = nullptr;
  std::vector<const bf16*> w;   // [L][9]
  std::vector<int> X;
  int N = 0;
  dex_decode_cfg cfg = {};
  cudaStream_t st = nullptr;
  int n_sm = 0;
  int gemm_ctas = 0;           // persistent GEMM grid (CTAs per SM x SMs), fixed per handle
  // k segments per tile of each weight shape (fixed per handle: results depend on them)
  int seg_qkv = 1, seg_o = 1, seg_gu = 1, seg_d = 1, seg_lm = 1;
  size_t partial_bytes = 0;    // segment-partial workspace
  // inducing adapters of the non-final depths (Appendix C.2), n_adapters = N - 1 or 0
  int n_adapters = 0, seg_ad1 = 1, seg_ad2 = 1;
  std::vector<const bf16*> ad_g, ad_b1, ad_b2;
  std::vector<float> ad_alpha;
  std::vector<const uint8_t*> pk_ad1, pk_ad2;   // packed W1 [2d][d], W2 [d][2d]
  bf16* ad_act = nullptr;                        // [2][rows_cap][2d] hidden activations
  CUtensorMap tm_adact[17];
  size_t gemm_smem = 0;        // shared-memory budget of a small-tile GEMM CTA
  std::unique_ptr<dex::Lattice> lat, lat_ar;
  std::vector<int> mode;                 // per sequence: 0 idle, 1 DEX, 2 AR
  std::vector<int> n_done;
  std::vector<dex_copy_job> pending_jobs, pending_jobs_ar;
  int rows_cap = 0, n_slots = 0, max_groups = 0, hrows = 0;
  // device buffers
  std::vector<void*> allocs;
  __half *kv_commit = nullptr, *kv_pool = nullptr;   // fp16 K/V caches
  CUtensorMap tm_kv;                                 // committed cache rows for the attention
  // activation buffers: two planes of rows_cap rows each, hi then lo (x ~= hi + lo)
  bf16 *hb = nullptr, *exit_hb = nullptr, *attn_out = nullptr, *act = nullptr;
  float *hidden = nullptr, *ssq = nullptr, *exit_ssq = nullptr, *q = nullptr, *partial = nullptr,
        *attn_part = nullptr, *logits_dbg = nullptr;
  int32_t *counters = nullptr, *attn_counters = nullptr, *err = nullptr;
  long long* acc64 = nullptr;   // fixed-point split-K tile sums (zero at rest)
  bool red_sum = false;          // layer GEMMs of decode rounds sum k segments at L2 in fixed point
  size_t acc_bytes = 0, counter_bytes = 0, attn_counter_bytes = 0;
  float2* rope = nullptr;
  unsigned long long* best = nullptr;
  const bf16** d_attn_norms = nullptr;
  uint8_t* d_plan = nullptr;
  size_t plan_cap = 0;
  // pinned host
  uint8_t* h_plan = nullptr;
  // pinned copy of the device flag + best keys: [0..1] the error flag, [2 ..] best keys
  unsigned long long* h_best = nullptr;
  // packed GEMM weights (one swizzled 16 KB box per (tile, k-block), tile-major)
  std::vector<const uint8_t*> pk_qkv, pk_o, pk_gu, pk_d;
  const uint8_t* pk_lm = nullptr;
  size_t packed_total = 0;
  // tensor maps
  std::vector<CUtensorMap> tm_q, tm_k, tm_v, tm_o, tm_g, tm_u, tm_d;
  CUtensorMap tm_lm;
  CUtensorMap tm_hb[17], tm_attn[17], tm_act[17], tm_exit[17];
  // bookkeeping
  dex_stats stats = {};
  int timing = 0;
  std::vector<dex_plan_node> last_plan;
  std::vector<int32_t> last_tokens;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> gemm_events;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> attn_events;
  bool broken = false;
  // GEMM timeline diagnostics (timing level 3 with DEX_TIMELINE set)
  unsigned long long* timeline = nullptr;
  int tl_cap = 0, tl_used = 0;
  std::vector<int32_t> tl_meta;   // per launch: epi, n_groups, nt, n_tiles, n_segs, kblocks, n_ctas, rows
  unsigned long long* atl = nullptr;   // attention records (same level and file, suffix ".attn")
  int atl_cap = 0, atl_used = 0;
  std::vector<int32_t> atl_meta;       // per launch: n_items, n_units, grid
  // host-side allocation-failure injection (DEX_FAIL_ALLOC_AT=k: the k-th allocation of
  // dex_init fails), for tests of the DEX_ENOMEM path
  int alloc_fail_at = 0, alloc_count = 0;
  int prefill_rows = kPrefillRowsMax;   // prompt positions per prefill pass
  int prefill_group_rows = 64;   // node rows per GEMM group of a prefill pass (the node tile)
  std::map<std::pair<int, int>, int> prefill_segs;   // (tiles of a launch, k-blocks) -> segments

  // Releases everything the handle owns; runs on dex_free and on every failing dex_init.
  ~dex_handle() {
    cudaStreamSynchronize(st);
    for (void* p : allocs) cudaFree(p);
    if (h_plan) cudaFreeHost(h_plan);
    if (h_best) cudaFreeHost(h_best);
    for (auto e : ev_pool) cudaEventDestroy(e);
  }
};

namespace {

bool debug_enabled() {
  static const bool on = getenv("DEX_DEBUG") != nullptr;
  return on;
}

int cuda_fail(dex_handle* h, cudaError_t e) {
  if (e == cudaSuccess) return DEX_OK;
  if (debug_enabled()) fprintf(stderr, "dex: CUDA error %s (%s)\n", cudaGetErrorName(e), cudaGetErrorString(e));
  if (h) h->broken = true;
  return DEX_ECUDA;
}

bool injected_alloc_failure(dex_handle* h) {
  return h->alloc_fail_at > 0 && ++h->alloc_count == h->alloc_fail_at;
}

template <typename T>
int dalloc(dex_handle* h, T** p, size_t bytes) {
  void* v = nullptr;
  if (injected_alloc_failure(h) || cudaMalloc(&v, bytes ? bytes : 16) != cudaSuccess) return DEX_ENOMEM;
  h->allocs.push_back(v);
  *p = reinterpret_cast<T*>(v);
  return DEX_OK;
}

template <typename T>
int halloc(dex_handle* h, T** p, size_t bytes) {   // pinned host memory, freed by the handle
  void* v = nullptr;
  if (injected_alloc_failure(h) || cudaMallocHost(&v, bytes ? bytes : 16) != cudaSuccess) return DEX_ENOMEM;
  *p = reinterpret_cast<T*>(v);
  return DEX_OK;
}

cudaEvent_t next_event(dex_handle* h) {
  if (h->ev_used == h->ev_pool.size()) {
    cudaEvent_t e;
    cudaEventCreate(&e);
    h->ev_pool.push_back(e);
  }
  return h->ev_pool[h->ev_used++];
}

const bf16* W(const dex_handle* h, int layer, int j) { return h->w[static_cast<size_t>(layer) * 9 + j]; }

// Per-round description of the node batch, built on the host and uploaded once.
struct RoundTables {
  std::vector<dex::DevNode> nodes;
  std::vector<int32_t> tails, priors;
  std::vector<dex::AttnItem> items;     // attention items of every layer slot, slot after slot
  std::vector<dex_copy_job> jobs;
};

// A batch of node rows that runs a contiguous range of layers: one stage of a DEX round,
// or a prefill chunk.  `items` are its attention items (layer filled in per slot).
struct Batch {
  int off, n, l0, l1;
  int stage = -1;   // lattice stage of a DEX round's batch (-1: prefill)
  std::vector<dex::AttnItem> items;
};

// Layer slot j of a round: layer l0 + j of every batch that has it, run as one grouped
// launch per operator.  Batches of a round are independent (their inputs come from the
// previous round), so their layers may share launches.
struct Slot {
  std::vector<int> batch;   // batch indices
  int item0 = 0, n_items = 0, n_units = 0, max_groups = 1, max_rows = 1;
};

std::vector<Slot> build_slots(const std::vector<Batch>& batches, int kvh, RoundTables* t) {
  int max_len = 0;
  for (const auto& b : batches) max_len = std::max(max_len, b.l1 - b.l0);
  std::vector<Slot> slots(max_len);
  for (int j = 0; j < max_len; ++j) {
    Slot& sl = slots[j];
    sl.item0 = static_cast<int>(t->items.size());
    for (size_t bi = 0; bi < batches.size(); ++bi) {
      const Batch& b = batches[bi];
      if (b.l0 + j >= b.l1 || b.n == 0) continue;
      sl.batch.push_back(static_cast<int>(bi));
      for (dex::AttnItem it : b.items) {
        it.layer = b.l0 + j;
        it.counter = sl.n_items++;
        it.unit0 = sl.n_units;
        sl.n_units += kvh * it.n_groups;
        sl.max_groups = std::max(sl.max_groups, it.n_groups);
        sl.max_rows = std::max(sl.max_rows, it.row_end - it.row_begin);
        t->items.push_back(it);
      }
    }
  }
  return slots;
}

struct Uploaded {
  dex::DevNode* nodes;
  int32_t *tails, *priors;
  dex::AttnItem* items;
  dex::CopyJob* jobs;
};

int upload(dex_handle* h, const RoundTables& t, Uploaded* u) {
  size_t off = 0;
  auto place = [&](size_t bytes) {
    size_t o = (off + 255) & ~size_t(255);
    off = o + bytes;
    return o;
  };
  const size_t o_nodes = place(t.nodes.size() * sizeof(dex::DevNode));
  const size_t o_tails = place(t.tails.size() * 4 + 4);
  const size_t o_priors = place(t.priors.size() * 4 + 4);
  const size_t o_items = place(t.items.size() * sizeof(dex::AttnItem));
  const size_t o_jobs = place(t.jobs.size() * sizeof(dex::CopyJob));
  if (off > h->plan_cap) return DEX_ECAPACITY;
  memcpy(h->h_plan + o_nodes, t.nodes.data(), t.nodes.size() * sizeof(dex::DevNode));
  memcpy(h->h_plan + o_tails, t.tails.data(), t.tails.size() * 4);
  memcpy(h->h_plan + o_priors, t.priors.data(), t.priors.size() * 4);
  memcpy(h->h_plan + o_items, t.items.data(), t.items.size() * sizeof(dex::AttnItem));
  memcpy(h->h_plan + o_jobs, t.jobs.data(), t.jobs.size() * sizeof(dex::CopyJob));
  if (cudaMemcpyAsync(h->d_plan, h->h_plan, off, cudaMemcpyHostToDevice, h->st) != cudaSuccess)
    return cuda_fail(h, cudaGetLastError());
  h->stats.h2d_bytes += static_cast<int64_t>(off);
  u->nodes = reinterpret_cast<dex::DevNode*>(h->d_plan + o_nodes);
  u->tails = reinterpret_cast<int32_t*>(h->d_plan + o_tails);
  u->priors = reinterpret_cast<int32_t*>(h->d_plan + o_priors);
  u->items = reinterpret_cast<dex::AttnItem*>(h->d_plan + o_items);
  u->jobs = reinterpret_cast<dex::CopyJob*>(h->d_plan + o_jobs);
  return DEX_OK;
}

dex::GemmArgs base_args(dex_handle* h) {
  dex::GemmArgs a = {};
  a.err = h->err;
  a.d = h->d;
  a.H = h->H;
  a.KVH = h->KVH;
  a.hd = h->hd;
  a.L = h->L;
  a.d_ff = h->dff;
  a.vocab = h->V;
  a.max_ctx = h->cfg.max_ctx;
  a.n_slots = h->n_slots;
  a.eps = h->eps;
  a.partial = h->partial;
  a.counters = h->counters;
  a.evict_first = 1;
  a.plane_rows = h->rows_cap;
  return a;
}

// Launch one grouped GEMM.  Every group has at most 256 node rows; nmax is the largest.
int gemm(dex_handle* h, int epi, const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& a2,
         const CUtensorMap* bmaps, dex::GemmArgs a, int nmax, int64_t weight_bytes, int64_t act_bytes_per_row,
         bool layer_gemm = false, size_t smem_budget = 0) {
  if (nmax < 1 || nmax > 256) return DEX_ECAPACITY;
  a.nt = (nmax + 15) & ~15;
  a.n_ctas = h->gemm_ctas;
  if (a.n_segs > 1 &&
      dex::gemm_partial_bytes(a.nt, static_cast<size_t>(a.n_groups) * a.n_tiles * a.n_segs) > h->partial_bytes)
    return DEX_ECAPACITY;
  a.tmem_cols = pow2_at_least(a.nt);
  a.stages = dex::gemm_stages_for(a.nt, epi, h->gemm_smem);
  if (smem_budget) {   // a fixed budget for every node tile (two CTAs per SM), when two stages fit it
    int st = 8;
    while (st > 2 && dex::gemm_smem_bytes(a.nt, st, epi) > smem_budget) --st;
    if (dex::gemm_smem_bytes(a.nt, st, epi) <= smem_budget) a.stages = st;
  }
  // A decoder whose lattice gives a sequence at most 16 nodes per round sums the k segments
  // of its layer GEMMs at L2 in fixed point (no partial tiles to read back at the end of a
  // launch); one with a wider lattice, the exit head, the adapters and prefill passes sum
  // fp32 partial tiles in segment order.  The choice depends on the exploration set only,
  // so a node's result is the same whatever its round, batch or launch.
  a.acc = h->acc64;
  a.sum_mode = (layer_gemm && h->red_sum) ? dex::SUM_FIXED_RED : dex::SUM_FP32;
  if (a.sum_mode == dex::SUM_FIXED_RED &&
      static_cast<size_t>(a.n_groups) * a.n_tiles * a.nt * 128 * sizeof(long long) > h->acc_bytes)
    return DEX_ECAPACITY;   // cannot happen: acc covers N groups of the widest round
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (h->timing == 2) {
    e0 = next_event(h);
    e1 = next_event(h);
    cudaEventRecord(e0, h->st);
  }
  if (h->timing == 3 && h->timeline && h->tl_used < h->tl_cap) {
    a.timeline = h->timeline + static_cast<size_t>(h->tl_used++) * h->gemm_ctas * dex::kTimelineSlots;
    int rows_all = 0;
    for (int g = 0; g < a.n_groups; ++g) rows_all += a.groups[g].n;
    const int32_t meta[8] = {epi, a.n_groups, a.nt, a.n_tiles, a.n_segs, a.kblocks, a.n_ctas, rows_all};
    h->tl_meta.insert(h->tl_meta.end(), meta, meta + 8);
  }
  cudaError_t e = dex::launch_gemm(epi, a0, a1, a2, bmaps[a.nt / 16], a, h->st, true);
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (h->timing == 2) {
    cudaEventRecord(e1, h->st);
    h->gemm_events.push_back({e0, e1});
  }
  int rows = 0;
  for (int g = 0; g < a.n_groups; ++g) rows += a.groups[g].n;
  h->stats.kernel_launches++;
  h->stats.gemm_launches++;
  h->stats.gemm_bytes += weight_bytes * a.n_groups + act_bytes_per_row * rows;
  return DEX_OK;
}

// Shared-memory budget of a prefill pass's GEMM CTAs: 113 KB keeps two CTAs per SM (228 KB
// per SM, 1 KB reserved per CTA) -- three ring stages at node tile 64, two at 128.
constexpr size_t kPrefillGemmSmem = 113 * 1024;

// The decoder layers of every slot: per slot, grouped QKV+RoPE+KV write, lattice
// attention, O + residual, gate/up + SwiGLU, down + residual over the slot's batches.
// Prefill passes (prefill = true) carry several node groups of the same layer per launch;
// their k segments follow the launch's own tile count (a prompt position's K/V may then
// differ in the last bits from what a decode round would write for it; DEX and plain AR
// decode from the same prefill, so their equality is unaffected), and the weights stay in
// L2 for the groups that read them after the first.
int run_layers(dex_handle* h, const Uploaded& u, const std::vector<Batch>& batches, const std::vector<Slot>& slots,
               bool with_exit, bool prefill = false) {
  const int qd = h->H * h->hd, kvd = h->KVH * h->hd;
  const int64_t d = h->d;
  auto segments = [&](int decode_segs, int n_tiles, int kblocks, int ng) {
    if (!prefill) return decode_segs;
    const std::pair<int, int> key(n_tiles * ng, kblocks);
    auto it = h->prefill_segs.find(key);
    if (it != h->prefill_segs.end()) return it->second;
    const int sg = dex::gemm_segments(n_tiles * ng, kblocks, h->gemm_ctas);
    h->prefill_segs[key] = sg;
    return sg;
  };
  for (size_t j = 0; j < slots.size(); ++j) {
    const Slot& sl = slots[j];
    const int ng = static_cast<int>(sl.batch.size());
    if (ng == 0) continue;
    int nmax = 0;
    for (int bi : sl.batch) nmax = std::max(nmax, batches[bi].n);
    auto fill_groups = [&](dex::GemmArgs& a, int op) {
      a.nodes = u.nodes;
      a.n_groups = ng;
      for (int g = 0; g < ng; ++g) {
        const Batch& b = batches[sl.batch[g]];
        const int l = b.l0 + static_cast<int>(j);
        dex::GemmGroup& gr = a.groups[g];
        gr = dex::GemmGroup{};
        gr.b_row0 = b.off;
        gr.n = b.n;
        gr.layer = l;
        if (op == 0) gr.a_packed = h->pk_qkv[l];
        if (op == 1) {
          gr.a_packed = h->pk_o[l];
          gr.has_next = 1;
          gr.g_next = W(h, l, 5);
        }
        if (op == 2) gr.a_packed = h->pk_gu[l];
        if (op == 3) {
          const bool last = (l == b.l1 - 1);
          gr.a_packed = h->pk_d[l];
          gr.has_next = (!last && l + 1 < h->L) ? 1 : 0;
          gr.g_next = (l + 1 < h->L) ? W(h, l + 1, 0) : nullptr;
          gr.stage_end = (last && with_exit) ? 1 : 0;
          if (gr.stage_end && b.stage >= 0 && b.stage < h->n_adapters) gr.g_exit = h->ad_g[b.stage];
        }
      }
    };
    const int l_first = batches[sl.batch[0]].l0 + static_cast<int>(j);   // tensor maps of one member (unused when packed)
    // QKV + RoPE + KV write
    dex::GemmArgs a = base_args(h);
    fill_groups(a, 0);
    a.kblocks = (h->d + 63) / 64;
    a.src_tiles0 = qd / 128;
    a.src_tiles1 = kvd / 128;
    a.n_tiles = (qd + 2 * kvd) / 128;
    a.n_segs = segments(h->seg_qkv, a.n_tiles, a.kblocks, ng);
    a.evict_first = prefill ? 0 : 1;
    a.ssq_in = h->ssq;
    a.q_out = h->q;
    a.kv_commit = h->kv_commit;
    a.kv_pool = h->kv_pool;
    a.rope = h->rope;
    int rc = gemm(h, dex::EPI_QKV, h->tm_q[l_first], h->tm_k[l_first], h->tm_v[l_first], h->tm_hb, a, nmax,
                  static_cast<int64_t>(qd + 2 * kvd) * d * 2, d * 4 + qd * 4 + 2 * kvd * 4, !prefill,
              prefill ? kPrefillGemmSmem : 0);
    if (rc) return rc;
    // lattice attention over every batch of the slot
    dex::AttnArgs at = {};
    at.nodes = u.nodes;
    at.items = u.items + sl.item0;
    at.n_items = sl.n_items;
    at.n_units = sl.n_units;
    at.tails = u.tails;
    at.q = h->q;
    at.kv_commit = h->kv_commit;
    at.kv_pool = h->kv_pool;
    at.out = h->attn_out;
    at.part = h->attn_part;
    at.counters = h->attn_counters;
    at.err = h->err;
    at.H = h->H;
    at.KVH = h->KVH;
    at.hd = h->hd;
    at.L = h->L;
    at.max_ctx = h->cfg.max_ctx;
    at.n_slots = h->n_slots;
    at.part_slots = h->max_groups + 1;
    at.plane_rows = h->rows_cap;
    at.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(h->hd)));
    at.early_kv = prefill ? 0 : 1;
    cudaEvent_t ae0 = nullptr, ae1 = nullptr;
    if (h->timing == 2) {
      ae0 = next_event(h);
      ae1 = next_event(h);
      cudaEventRecord(ae0, h->st);
    }
    if (h->timing == 3 && h->atl && h->atl_used < h->atl_cap) {
      at.timeline = h->atl + static_cast<size_t>(h->atl_used++) * h->n_sm * dex::kAttnTimelineSlots;
      const int32_t meta[3] = {sl.n_items, sl.n_units, std::min(h->n_sm, sl.n_units)};
      h->atl_meta.insert(h->atl_meta.end(), meta, meta + 3);
    }
    cudaError_t ce;
    if (prefill && dex::prefill_attention_supported(h->H, h->KVH, h->hd)) {
      // a prefill pass: consecutive positions of one sequence, rows 0 .. n-1 of the pass
      dex::PrefillAttnArgs pa = {};
      pa.nodes = u.nodes;
      for (int bi : sl.batch) pa.n_rows = std::max(pa.n_rows, batches[bi].off + batches[bi].n);
      pa.seq = batches[sl.batch[0]].items.empty() ? 0 : batches[sl.batch[0]].items[0].seq;
      pa.layer = batches[sl.batch[0]].l0 + static_cast<int>(j);
      pa.q = h->q;
      pa.out = h->attn_out;
      pa.plane_rows = h->rows_cap;
      pa.err = h->err;
      pa.H = h->H;
      pa.KVH = h->KVH;
      pa.hd = h->hd;
      pa.L = h->L;
      pa.max_ctx = h->cfg.max_ctx;
      pa.scale_log2 = at.scale_log2;
      ce = dex::launch_prefill_attention(h->tm_kv, pa, h->st, true);
    } else {
      ce = dex::launch_attention(h->tm_kv, at, h->n_sm, h->st, true);
    }
    if (ce != cudaSuccess) return cuda_fail(h, ce);
    if (h->timing == 2) {
      cudaEventRecord(ae1, h->st);
      h->attn_events.push_back({ae0, ae1});
    }
    h->stats.kernel_launches++;
    h->stats.attn_launches++;
    // O projection + residual
    a = base_args(h);
    fill_groups(a, 1);
    a.kblocks = (qd + 63) / 64;
    a.n_tiles = h->d / 128;
    a.n_segs = segments(h->seg_o, a.n_tiles, a.kblocks, ng);
    a.evict_first = prefill ? 0 : 1;
    a.src_tiles0 = a.n_tiles;
    a.hidden = h->hidden;
    a.hb_out = h->hb;
    a.ssq_out = h->ssq;
    rc = gemm(h, dex::EPI_RESID, h->tm_o[l_first], h->tm_o[l_first], h->tm_o[l_first], h->tm_attn, a, nmax,
              static_cast<int64_t>(qd) * d * 2, qd * 4 + d * 8 + d * 4, !prefill,
              prefill ? kPrefillGemmSmem : 0);
    if (rc) return rc;
    // gate/up + SwiGLU
    a = base_args(h);
    fill_groups(a, 2);
    a.kblocks = (h->d + 63) / 64;
    a.n_tiles = (h->dff + 63) / 64;
    a.n_segs = segments(h->seg_gu, a.n_tiles, a.kblocks, ng);
    a.evict_first = prefill ? 0 : 1;
    a.src_tiles0 = a.n_tiles;
    a.ssq_in = h->ssq;
    a.act_out = h->act;
    rc = gemm(h, dex::EPI_SWIGLU, h->tm_g[l_first], h->tm_u[l_first], h->tm_u[l_first], h->tm_hb, a, nmax,
              static_cast<int64_t>(2) * h->dff * d * 2, d * 4 + h->dff * 4, !prefill,
              prefill ? kPrefillGemmSmem : 0);
    if (rc) return rc;
    // down + residual (+ exit-head input at the stage boundary)
    a = base_args(h);
    fill_groups(a, 3);
    a.kblocks = (h->dff + 63) / 64;
    a.n_tiles = h->d / 128;
    a.n_segs = segments(h->seg_d, a.n_tiles, a.kblocks, ng);
    a.evict_first = prefill ? 0 : 1;
    a.src_tiles0 = a.n_tiles;
    a.hidden = h->hidden;
    a.hb_out = h->hb;
    a.ssq_out = h->ssq;
    a.exit_hb = h->exit_hb;
    a.g_final = h->final_norm;
    a.exit_ssq = h->exit_ssq;
    rc = gemm(h, dex::EPI_RESID, h->tm_d[l_first], h->tm_d[l_first], h->tm_d[l_first], h->tm_act, a, nmax,
              static_cast<int64_t>(h->dff) * d * 2, h->dff * 4 + d * 8 + d * 8, !prefill,
              prefill ? kPrefillGemmSmem : 0);
    if (rc) return rc;
  }
  return DEX_OK;
}

int check_device_error(dex_handle* h, int32_t flag) {
  if (flag == 0) return DEX_OK;
  if (debug_enabled()) fprintf(stderr, "dex: device error flag %d\n", flag);
  cudaMemsetAsync(h->err, 0, sizeof(int32_t), h->st);
  // a launch that gave up may leave arrival counters and tile sums away from zero
  cudaMemsetAsync(h->counters, 0, h->counter_bytes, h->st);
  cudaMemsetAsync(h->attn_counters, 0, h->attn_counter_bytes, h->st);
  cudaMemsetAsync(h->acc64, 0, h->acc_bytes, h->st);
  if (flag == dex::DEV_RANGE) return DEX_ERANGE;
  return flag == dex::DEV_BAD_INDEX ? DEX_ECUDA : DEX_ETIMEOUT;
}

// One round on lattice `lat` (DEX or the single-stage AR lattice).
int run_round(dex_handle* h, dex::Lattice* lat, std::vector<dex_copy_job>* pending, int32_t* out_tokens,
              int32_t* n_committed) {
  if (h->broken) return DEX_ECUDA;
  auto t_host0 = std::chrono::steady_clock::now();
  std::vector<dex_plan_node> plan;
  const int n = lat->plan(&plan);
  if (n < 0) return DEX_ECAPACITY;
  if (n == 0) return DEX_ESTATE;
  const int NS = lat->N();
  const std::vector<int>& X = lat->X();
  RoundTables t;
  std::vector<int> stage_off(NS + 1, 0);
  int max_stage = 0;
  for (const auto& p : plan) {
    if (p.target_pos >= h->cfg.max_ctx) return DEX_ECAPACITY;
    stage_off[p.stage + 1]++;
    max_stage = std::max(max_stage, p.stage);
  }
  for (int s = 0; s < NS; ++s) stage_off[s + 1] += stage_off[s];
  for (int k = 0; k < n; ++k) {
    const auto& p = plan[k];
    dex::DevNode dn = {};
    dn.seq = p.seq;
    dn.pos = p.pos;
    dn.c_end = p.c_end;
    dn.slot = p.slot;
    dn.hrow = p.seq * h->n_slots + p.slot;
    dn.kv_commit = p.kv_commit;
    dn.token = p.token;
    dn.first_layer = p.stage > 0 ? X[p.stage - 1] : 0;
    dn.tail_off = static_cast<int32_t>(t.tails.size());
    dn.n_tail = p.n_tail;
    for (int i = 0; i < p.n_tail; ++i) t.tails.push_back(p.tail[i]);
    dn.target_pos = p.target_pos;
    dn.unmasked = p.unmasked;
    dn.prior_off = static_cast<int32_t>(t.priors.size());
    dn.n_prior = p.n_prior;
    for (int i = 0; i < p.n_prior; ++i) t.priors.push_back(p.prior[i]);
    t.nodes.push_back(dn);
  }
  // one batch per live stage: its layers (d_{s-1}, d_s] and attention items over each
  // sequence's contiguous rows, at most one pass of queries per item (an item that fits one
  // pass takes the smaller single-pass attention CTA; the committed keys the items of a
  // sequence share are re-read from L2)
  const int rows_per_item = std::max(1, dex::kAttnPassQueries / (h->H / h->KVH));
  std::vector<Batch> batches;
  for (int s = 0; s <= max_stage; ++s) {
    Batch b;
    b.off = stage_off[s];
    b.n = stage_off[s + 1] - stage_off[s];
    b.l0 = s > 0 ? X[s - 1] : 0;
    b.l1 = X[s];
    b.stage = (NS == h->N) ? s : -1;   // adapters belong to the DEX lattice's stages only
    for (int k = b.off; k < b.off + b.n;) {
      int e = k;
      dex::AttnItem it = {};
      it.seq = plan[k].seq;
      it.row_begin = k;
      while (e < b.off + b.n && plan[e].seq == it.seq && e - k < rows_per_item) {
        it.max_pos = std::max(it.max_pos, plan[e].pos);
        it.max_cend = std::max(it.max_cend, plan[e].c_end);
        ++e;
      }
      it.row_end = e;
      it.n_groups = std::max(1, (dex::attn_bulk_end(it.max_pos) + dex::kAttnGroupPos - 1) / dex::kAttnGroupPos);
      b.items.push_back(it);
      k = e;
    }
    if (b.n > 256) return DEX_ECAPACITY;
    batches.push_back(b);
  }
  const std::vector<Slot> slots = build_slots(batches, h->KVH, &t);
  t.jobs = *pending;
  const double host_plan_ms =
      std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_host0).count();

  Uploaded u;
  int rc = upload(h, t, &u);
  if (rc) return rc;
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  if (h->timing >= 1)
    for (auto& e : ev) e = next_event(h);
  if (ev[0]) cudaEventRecord(ev[0], h->st);
  if (!t.jobs.empty()) {
    dex::CollapseArgs ca = {};
    ca.jobs = u.jobs;
    ca.n_jobs = static_cast<int>(t.jobs.size());
    ca.kv_commit = h->kv_commit;
    ca.kv_pool = h->kv_pool;
    ca.batch = h->cfg.batch;
    ca.err = h->err;
    ca.L = h->L;
    ca.KVH = h->KVH;
    ca.row_bytes = h->hd * 2;
    ca.max_ctx = h->cfg.max_ctx;
    ca.n_slots = h->n_slots;
    cudaError_t ce = dex::launch_collapse(ca, h->st, false);
    if (ce != cudaSuccess) return cuda_fail(h, ce);
    h->stats.kernel_launches++;
  }
  if (ev[1]) cudaEventRecord(ev[1], h->st);
  dex::AssembleArgs aa = {};
  aa.nodes = u.nodes;
  aa.n_rows = n;
  aa.d = h->d;
  aa.embed = h->embed;
  aa.attn_norm = h->d_attn_norms;
  aa.hidden = h->hidden;
  aa.hb = h->hb;
  aa.plane_rows = h->rows_cap;
  aa.ssq = h->ssq;
  aa.best = h->best;
  cudaError_t ce = dex::launch_assemble(aa, h->st, !t.jobs.empty());   // overlaps the collapse's tail
  if (ce != cudaSuccess) return cuda_fail(h, ce);
  h->stats.kernel_launches++;
  rc = run_layers(h, u, batches, slots, true);
  if (rc) return rc;
  // inducing adapters of the non-final stages: exit input h -> h + alpha (W2 SiLU(W1 n + b1) + b2)
  if (h->n_adapters > 0) {
    dex::GemmArgs up = base_args(h), dn = base_args(h);
    int ng = 0, nmax_ad = 0;
    for (const Batch& b : batches) {
      if (b.stage < 0 || b.stage >= h->n_adapters || b.n == 0) continue;
      dex::GemmGroup gu = {}, gd = {};
      gu.a_packed = h->pk_ad1[b.stage];
      gu.bias = h->ad_b1[b.stage];
      gd.a_packed = h->pk_ad2[b.stage];
      gd.bias = h->ad_b2[b.stage];
      gd.alpha = h->ad_alpha[b.stage];
      gu.b_row0 = gd.b_row0 = b.off;
      gu.n = gd.n = b.n;
      up.groups[ng] = gu;
      dn.groups[ng] = gd;
      ++ng;
      nmax_ad = std::max(nmax_ad, b.n);
    }
    if (ng > 0) {
      up.nodes = dn.nodes = u.nodes;
      up.n_groups = dn.n_groups = ng;
      up.kblocks = (h->d + 63) / 64;
      up.n_tiles = 2 * h->d / 128;
      up.n_segs = h->seg_ad1;
      up.src_tiles0 = up.n_tiles;
      up.ssq_in = h->exit_ssq;
      up.act_out = h->ad_act;
      up.d_ff = 2 * h->d;
      rc = gemm(h, dex::EPI_ADUP, h->tm_lm, h->tm_lm, h->tm_lm, h->tm_exit, up, nmax_ad,
                static_cast<int64_t>(2) * h->d * h->d * 2, static_cast<int64_t>(h->d) * 4 + 2 * h->d * 4);
      if (rc) return rc;
      dn.kblocks = (2 * h->d + 63) / 64;
      dn.n_tiles = h->d / 128;
      dn.n_segs = h->seg_ad2;
      dn.src_tiles0 = dn.n_tiles;
      dn.hidden = h->hidden;
      dn.exit_hb = h->exit_hb;
      dn.exit_ssq = h->exit_ssq;
      dn.g_final = h->final_norm;
      rc = gemm(h, dex::EPI_ADDOWN, h->tm_lm, h->tm_lm, h->tm_lm, h->tm_adact, dn, nmax_ad,
                static_cast<int64_t>(2) * h->d * h->d * 2, static_cast<int64_t>(2) * h->d * 4 + h->d * 8);
      if (rc) return rc;
      h->stats.weight_bytes += static_cast<int64_t>(ng) * 8 * h->d * h->d;
    }
  }
  if (ev[2]) cudaEventRecord(ev[2], h->st);
  // exit head + DECS over every node of the round
  {
    dex::GemmArgs a = base_args(h);
    a.nodes = u.nodes;
    a.kblocks = (h->d + 63) / 64;
    a.n_tiles = (h->V + 127) / 128;
    a.n_segs = h->seg_lm;
    a.src_tiles0 = a.n_tiles;
    a.ssq_in = h->exit_ssq;
    a.logits_dbg = h->cfg.debug_logits ? h->logits_dbg : nullptr;
    a.best = h->best;
    a.priors = u.priors;
    a.sample = h->cfg.sample;
    a.tau = h->cfg.tau;
    a.seed = h->cfg.seed;
    for (int r0 = 0; r0 < n && !rc; r0 += 256) {
      a.n_groups = 1;
      a.groups[0] = dex::GemmGroup{};
      a.groups[0].a_packed = h->pk_lm;
      a.groups[0].b_row0 = r0;
      a.groups[0].n = std::min(256, n - r0);
      rc = gemm(h, dex::EPI_EXIT, h->tm_lm, h->tm_lm, h->tm_lm, h->tm_exit, a, a.groups[0].n,
                static_cast<int64_t>(h->V) * h->d * 2, static_cast<int64_t>(h->d) * 4);
    }
    if (rc) return rc;
  }
  if (ev[3]) cudaEventRecord(ev[3], h->st);
  // tokens (and the device error flag) back to the host: the round's only sync
  if (cudaMemcpyAsync(h->h_best, h->err, (n + 2) * sizeof(unsigned long long), cudaMemcpyDeviceToHost, h->st) !=
      cudaSuccess)
    return cuda_fail(h, cudaGetLastError());
  if (cudaStreamSynchronize(h->st) != cudaSuccess) return cuda_fail(h, cudaGetLastError());
  h->stats.d2h_bytes += (n + 2) * 8;
  const int32_t dev_err = static_cast<int32_t>(h->h_best[0] & 0xffffffffull);
  if (dev_err) return check_device_error(h, dev_err);
  auto t_host1 = std::chrono::steady_clock::now();
  std::vector<int32_t> tokens(n);
  for (int k = 0; k < n; ++k) tokens[k] = static_cast<int32_t>(~static_cast<uint32_t>(h->h_best[2 + k] & 0xffffffffull));
  std::vector<int32_t> committed(lat->batch()), kstar(lat->batch());
  lat->update(plan, tokens.data(), committed.data(), kstar.data(), pending);
  // statistics
  h->stats.rounds++;
  h->stats.nodes += n;
  h->stats.max_round_nodes = std::max<int64_t>(h->stats.max_round_nodes, n);
  h->stats.layer_passes += X[max_stage];
  const int64_t layer_w = (static_cast<int64_t>(h->H + 2 * h->KVH) * h->hd * h->d + static_cast<int64_t>(h->H) *
                           h->hd * h->d + 3ll * h->dff * h->d) * 2;
  h->stats.weight_bytes += layer_w * X[max_stage] + static_cast<int64_t>(h->V) * h->d * 2;
  const int64_t kv_row = 2ll * h->KVH * h->hd * 2;   // fp16 K and V of one position and layer
  for (const Batch& b : batches) {
    const int nl = b.l1 - b.l0;
    // committed keys and values once per (sequence, layer), however many items read them
    for (size_t i = 0; i < b.items.size(); ++i) {
      int cend = b.items[i].max_cend;
      while (i + 1 < b.items.size() && b.items[i + 1].seq == b.items[i].seq) cend = std::max(cend, b.items[++i].max_cend);
      h->stats.kv_bytes += kv_row * nl * cend;
    }
    for (int k = b.off; k < b.off + b.n; ++k) {
      h->stats.node_layers += nl;
      h->stats.kv_bytes += kv_row * nl * plan[k].n_tail;
    }
  }
  for (int b = 0; b < lat->batch(); ++b) {
    out_tokens[b] = committed[b] >= 0 ? committed[b] : -1;
    n_committed[b] = committed[b] >= 0 ? 1 : 0;
    if (committed[b] >= 0) {
      h->stats.commits++;
      h->stats.depth_charge += X[kstar[b]];
      h->stats.kstar_hist[std::min(kstar[b], 15)]++;
      if (++h->n_done[b] >= h->cfg.max_new) lat->stop(b);
    }
  }
  h->last_plan = plan;
  h->last_tokens = tokens;
  const double host_upd_ms =
      std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_host1).count();
  h->stats.ms_host += host_plan_ms + host_upd_ms;
  if (h->timing >= 1) {
    float ms;
    cudaEventElapsedTime(&ms, ev[0], ev[1]);
    h->stats.ms_collapse += ms;
    cudaEventElapsedTime(&ms, ev[1], ev[2]);
    h->stats.ms_expand += ms;
    cudaEventElapsedTime(&ms, ev[2], ev[3]);
    h->stats.ms_exit += ms;
  }
  if (h->timing == 2) {
    for (auto& pr : h->gemm_events) {
      float ms;
      cudaEventElapsedTime(&ms, pr.first, pr.second);
      h->stats.ms_gemm += ms;
    }
  }
  if (h->timing == 2) {
    for (auto& pr : h->attn_events) {
      float ms;
      cudaEventElapsedTime(&ms, pr.first, pr.second);
      h->stats.ms_attn += ms;
    }
  }
  h->gemm_events.clear();
  h->attn_events.clear();
  h->ev_used = 0;
  return DEX_OK;
}

}  // namespace

extern "C" {

const char* dex_strerror(int code) {
  switch (code) {
    case DEX_OK: return "ok";
    case DEX_EINVAL: return "invalid argument";
    case DEX_ENOMEM: return "out of memory";
    case DEX_ECUDA: return "CUDA error";
    case DEX_ECAPACITY: return "capacity exceeded (max_ctx / max_new / lattice size)";
    case DEX_ETIMEOUT: return "a bounded device wait timed out";
    case DEX_ESTATE: return "call out of order";
    case DEX_ENODEV: return "no sm_103 device";
    case DEX_ERANGE: return "a split-K partial sum outside the fixed-point range (not finite or >= 2^30)";
    default: return "unknown error";
  }
}

// Diagnostics file of timing level 3: int64 header {launches, n_ctas, slots}, then int32
// metadata [launches][8], then the uint64 records [launches][n_ctas][slots].
static void write_attn_timeline(dex_handle* h, const char* path) {
  if (!h->atl || h->atl_used == 0) return;
  const size_t words = static_cast<size_t>(h->atl_used) * h->n_sm * dex::kAttnTimelineSlots;
  std::vector<unsigned long long> buf(words);
  if (cudaMemcpy(buf.data(), h->atl, words * 8, cudaMemcpyDeviceToHost) != cudaSuccess) return;
  const std::string p = std::string(path) + ".attn";
  FILE* f = fopen(p.c_str(), "wb");
  if (!f) return;
  const int64_t hdr[3] = {h->atl_used, h->n_sm, dex::kAttnTimelineSlots};
  fwrite(hdr, sizeof(hdr), 1, f);
  fwrite(h->atl_meta.data(), 4, h->atl_meta.size(), f);
  fwrite(buf.data(), 8, words, f);
  fclose(f);
}

static void write_timeline(dex_handle* h) {
  const char* path = getenv("DEX_TIMELINE");
  if (path) write_attn_timeline(h, path);
  if (!path || !h->timeline || h->tl_used == 0) return;
  const size_t words = static_cast<size_t>(h->tl_used) * h->gemm_ctas * dex::kTimelineSlots;
  std::vector<unsigned long long> buf(words);
  if (cudaMemcpy(buf.data(), h->timeline, words * 8, cudaMemcpyDeviceToHost) != cudaSuccess) return;
  FILE* f = fopen(path, "wb");
  if (!f) return;
  const int64_t hdr[3] = {h->tl_used, h->gemm_ctas, dex::kTimelineSlots};
  fwrite(hdr, sizeof(hdr), 1, f);
  fwrite(h->tl_meta.data(), 4, h->tl_meta.size(), f);
  fwrite(buf.data(), 8, words, f);
  fclose(f);
}

void dex_free(dex_handle* h) {
  if (!h) return;
  cudaStreamSynchronize(h->st);
  write_timeline(h);
  delete h;   // the destructor releases device, pinned and event resources
}

int dex_init(const dex_model* m, const int32_t* X, int32_t n_X, const dex_decode_cfg* cfg, void* stream,
             dex_handle** out) {
  if (!m || !X || !cfg || !out) return DEX_EINVAL;
  *out = nullptr;
  if (m->n_layers < 1 || m->d_model % 128 || m->d_model > 8192 || (m->head_dim != 64 && m->head_dim != 128) || m->n_kv_heads < 1 ||
      m->n_heads % m->n_kv_heads || (m->n_heads * m->head_dim) % 128 || (m->n_kv_heads * m->head_dim) % 128 ||
      m->d_ff < 64 || m->d_ff % 8 || m->vocab < 2 || !m->embed || !m->final_norm || !m->lm_head || !m->layers)
    return DEX_EINVAL;
  static_assert(dex::kAttnWindow > 10, "the attention window must cover every node's branch keys (|X| <= 10)");
  if (n_X < 1 || n_X > 10 || X[n_X - 1] != m->n_layers) return DEX_EINVAL;
  for (int i = 0; i < n_X; ++i)
    if (X[i] < 1 || (i > 0 && X[i] <= X[i - 1])) return DEX_EINVAL;
  if (cfg->batch < 1 || cfg->batch > 64 || cfg->max_ctx < 2 || cfg->max_ctx > 4096 || cfg->max_new < 1 ||
      (cfg->sample && !(cfg->tau > 0)) || cfg->max_branch < 0)
    return DEX_EINVAL;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DEX_ENODEV;
  if (prop.major != 10 || prop.minor != 3) return DEX_ENODEV;
  if (get_encoder()) return DEX_ECUDA;

  std::unique_ptr<dex_handle> hp(new (std::nothrow) dex_handle());
  if (!hp) return DEX_ENOMEM;
  dex_handle* h = hp.get();
  h->L = m->n_layers;
  h->d = m->d_model;
  h->H = m->n_heads;
  h->KVH = m->n_kv_heads;
  h->hd = m->head_dim;
  h->dff = m->d_ff;
  h->V = m->vocab;
  h->eps = m->rms_eps;
  h->theta = m->rope_theta;
  h->embed = static_cast<const bf16*>(m->embed);
  h->final_norm = static_cast<const bf16*>(m->final_norm);
  h->lm_head = static_cast<const bf16*>(m->lm_head);
  h->w.resize(static_cast<size_t>(h->L) * 9);
  for (size_t i = 0; i < h->w.size(); ++i) {
    h->w[i] = static_cast<const bf16*>(m->layers[i]);
    if (!h->w[i]) return DEX_EINVAL;
  }
  h->X.assign(X, X + n_X);
  h->N = n_X;
  if (m->adapters && n_X > 1) {   // one adapter per non-final depth
    if (!m->adapter_alpha) return DEX_EINVAL;
    h->n_adapters = n_X - 1;
    for (int k = 0; k < h->n_adapters; ++k) {
      const void* const* ap = m->adapters + static_cast<size_t>(k) * 5;
      for (int j = 0; j < 5; ++j)
        if (!ap[j] || (reinterpret_cast<uintptr_t>(ap[j]) & 15)) return DEX_EINVAL;
      h->ad_g.push_back(static_cast<const bf16*>(ap[0]));
      h->ad_b1.push_back(static_cast<const bf16*>(ap[2]));
      h->ad_b2.push_back(static_cast<const bf16*>(ap[4]));
      h->ad_alpha.push_back(m->adapter_alpha[k]);
    }
  }
  h->cfg = *cfg;
  h->st = static_cast<cudaStream_t>(stream);
  if (const char* f = getenv("DEX_FAIL_ALLOC_AT")) h->alloc_fail_at = atoi(f);
  h->n_sm = prop.multiProcessorCount;
  // GEMM launch shape (tunable for experiments; the partition, hence every result,
  // depends on it, so it is fixed for the handle's lifetime)
  {
    const char* c = getenv("DEX_GEMM_CTAS_PER_SM");
    const char* m = getenv("DEX_GEMM_SMEM_KB");
    const int cps = c ? atoi(c) : 2;
    const int kb = m ? atoi(m) : 104;
    if (cps < 1 || cps > 4 || kb < 32 || kb > 227) return DEX_EINVAL;
    h->gemm_ctas = h->n_sm * cps;
    h->gemm_smem = static_cast<size_t>(kb) * 1024;
    // prompt positions per prefill pass (a multiple of 16 in [16, kPrefillRowsMax]) and node
    // rows per GEMM group of a pass (a multiple of 16 in [16, 256]), at most kMaxGroups groups
    if (const char* pr = getenv("DEX_PREFILL_ROWS")) h->prefill_rows = atoi(pr);
    if (const char* pg = getenv("DEX_PREFILL_GROUP_ROWS")) h->prefill_group_rows = atoi(pg);
    if (h->prefill_rows < 16 || h->prefill_rows > kPrefillRowsMax || (h->prefill_rows & 15) ||
        h->prefill_group_rows < 16 || h->prefill_group_rows > 256 || (h->prefill_group_rows & 15))
      return DEX_EINVAL;
    if ((h->prefill_rows + h->prefill_group_rows - 1) / h->prefill_group_rows > dex::kMaxGroups) return DEX_EINVAL;
  }
  h->lat.reset(new dex::Lattice(X, n_X, cfg->batch, cfg->decs != 0, cfg->max_branch));
  const int32_t XL[1] = {h->L};
  h->lat_ar.reset(new dex::Lattice(XL, 1, cfg->batch, false));
  h->mode.assign(cfg->batch, 0);
  h->n_done.assign(cfg->batch, 0);
  h->n_slots = h->lat->n_slots();
  h->rows_cap = std::max(h->lat->max_round_nodes(), kPrefillRowsMax);
  h->max_groups = (cfg->max_ctx + dex::kAttnGroupPos - 1) / dex::kAttnGroupPos;
  h->hrows = cfg->batch * h->n_slots + kPrefillRowsMax;

  const size_t B = cfg->batch, L = h->L, KVH = h->KVH, hd = h->hd, ctx = cfg->max_ctx, R = h->rows_cap;
  if (B * L * 2 * KVH * ctx >= (size_t(1) << 31)) return DEX_ECAPACITY;   // committed rows: 32-bit TMA rows
  const int qd = h->H * h->hd, kvd = h->KVH * h->hd;
  int rc = 0;
  rc |= dalloc(h, &h->kv_commit, B * L * 2 * KVH * ctx * hd * 2);
  rc |= dalloc(h, &h->kv_pool, B * h->n_slots * L * 2 * KVH * hd * 2);
  rc |= dalloc(h, &h->hidden, static_cast<size_t>(h->hrows) * h->d * 4);
  rc |= dalloc(h, &h->hb, 2 * R * h->d * 2);
  rc |= dalloc(h, &h->exit_hb, 2 * R * h->d * 2);
  rc |= dalloc(h, &h->attn_out, 2 * R * qd * 2);
  rc |= dalloc(h, &h->act, 2 * R * h->dff * 2);
  if (h->n_adapters) rc |= dalloc(h, &h->ad_act, 2 * R * 2 * static_cast<size_t>(h->d) * 2);
  rc |= dalloc(h, &h->ssq, R * (h->d / 128) * 4);
  rc |= dalloc(h, &h->exit_ssq, R * (h->d / 128) * 4);
  rc |= dalloc(h, &h->q, R * qd * 4);
  rc |= dalloc(h, &h->attn_part, R * h->H * (h->max_groups + 1) * (hd + 2) * 4);
  rc |= dalloc(h, &h->attn_counters, (static_cast<size_t>(B) * h->N + R) * KVH * 4);
  rc |= dalloc(h, &h->rope, ctx * (hd / 2) * sizeof(float2));
  // the device error flag (16 bytes), then the best keys [R]: one copy of the first n + 2
  // words per round brings the flag and the round's tokens back together
  {
    unsigned long long* base = nullptr;
    rc |= dalloc(h, &base, (R + 2) * 8);
    if (base) {
      h->err = reinterpret_cast<int32_t*>(base);
      h->best = base + 2;
    }
  }
  rc |= dalloc(h, &h->d_attn_norms, L * sizeof(void*));
  if (cfg->debug_logits) rc |= dalloc(h, &h->logits_dbg, R * static_cast<size_t>(h->V) * 4);
  if (rc) return DEX_ENOMEM;
  // partial-tile workspace of the persistent GEMM (two slots per CTA) and per-tile counters
  const size_t ntiles_max = std::max<size_t>({static_cast<size_t>((qd + 2 * kvd) / 128),
                                              static_cast<size_t>(h->d / 128),
                                              static_cast<size_t>((h->dff + 63) / 64),
                                              static_cast<size_t>((h->V + 127) / 128)});
  // fixed k segments per weight shape, and a partial workspace for the largest launch:
  // a prefill chunk (one group, node tile 256) or a round (N groups, node tile <= rows)
  {
    const int kb_d = (h->d + 63) / 64, kb_q = (qd + 63) / 64, kb_f = (h->dff + 63) / 64;
    const int t_qkv = (qd + 2 * kvd) / 128, t_o = h->d / 128, t_gu = (h->dff + 63) / 64, t_lm = (h->V + 127) / 128;
    h->seg_qkv = dex::gemm_segments(t_qkv, kb_d, h->gemm_ctas);
    h->seg_o = dex::gemm_segments(t_o, kb_q, h->gemm_ctas);
    h->seg_gu = dex::gemm_segments(t_gu, kb_d, h->gemm_ctas);
    h->seg_d = dex::gemm_segments(t_o, kb_f, h->gemm_ctas);
    h->seg_lm = dex::gemm_segments(t_lm, kb_d, h->gemm_ctas);
    h->seg_ad1 = dex::gemm_segments(2 * h->d / 128, kb_d, h->gemm_ctas);
    h->seg_ad2 = dex::gemm_segments(t_o, (2 * h->d + 63) / 64, h->gemm_ctas);
    const size_t u_layer = std::max<size_t>({static_cast<size_t>(t_qkv) * h->seg_qkv,
                                            static_cast<size_t>(t_o) * h->seg_o,
                                            static_cast<size_t>(t_gu) * h->seg_gu,
                                            static_cast<size_t>(t_o) * h->seg_d,
                                            static_cast<size_t>(2 * h->d / 128) * h->seg_ad1,
                                            static_cast<size_t>(t_o) * h->seg_ad2});
    const int nt_round = std::min(256, (std::max(1, h->lat->max_round_nodes()) + 15) & ~15);
    h->partial_bytes = std::max({dex::gemm_partial_bytes(nt_round, u_layer * std::max(1, h->N)),
                                 dex::gemm_partial_bytes(256, static_cast<size_t>(t_lm) * h->seg_lm)});
    // prefill passes: 1..ng_max groups of prefill_group_rows rows, their own segment counts
    const int ng_max = (h->prefill_rows + h->prefill_group_rows - 1) / h->prefill_group_rows;
    const std::pair<int, int> ops[4] = {{t_qkv, kb_d}, {t_o, kb_q}, {t_gu, kb_d}, {t_o, kb_f}};
    for (int ng = 1; ng <= ng_max; ++ng)
      for (const auto& op : ops) {
        const int sg = dex::gemm_segments(op.first * ng, op.second, h->gemm_ctas);
        h->prefill_segs[std::make_pair(op.first * ng, op.second)] = sg;
        h->partial_bytes = std::max(h->partial_bytes,
                                    dex::gemm_partial_bytes(h->prefill_group_rows, static_cast<size_t>(op.first) * ng * sg));
      }
    // fixed-point tile sums of the layer launches (at most N groups of the widest round) when
    // a sequence's round holds at most 16 nodes (2^(N-1) <= 16); DEX_SUM_FP32=1 keeps fp32
    // partial tiles for every decoder
    const char* fp32_only = getenv("DEX_SUM_FP32");
    h->red_sum = h->N <= 5 && !(fp32_only && atoi(fp32_only) != 0);
    const size_t t_layer = std::max<size_t>({static_cast<size_t>(t_qkv), static_cast<size_t>(t_o),
                                             static_cast<size_t>(t_gu)});
    h->acc_bytes = h->red_sum ? static_cast<size_t>(std::max(1, h->N)) * t_layer * nt_round * 128 * sizeof(long long)
                              : 16;
    if (debug_enabled())
      fprintf(stderr, "dex: segments qkv %d o %d gu %d down %d lm %d, partial workspace %.1f MB, %s layer sums\n",
              h->seg_qkv, h->seg_o, h->seg_gu, h->seg_d, h->seg_lm, h->partial_bytes / 1e6,
              h->red_sum ? "fixed-point (L2)" : "fp32 partial");
  }
  // arrival counters: one per (group, tile) of a launch, up to kMaxGroups groups
  h->counter_bytes = ntiles_max * 4 * std::max(dex::kMaxGroups, h->N);
  h->attn_counter_bytes = (static_cast<size_t>(B) * h->N + R) * KVH * 4;
  if (dalloc(h, &h->partial, h->partial_bytes) || dalloc(h, &h->counters, h->counter_bytes) ||
      dalloc(h, &h->acc64, h->acc_bytes))
    return DEX_ENOMEM;
  h->plan_cap = (R * sizeof(dex::DevNode) + R * 16 * 8 +
                 static_cast<size_t>(L) * (B * h->N + R + 8) * sizeof(dex::AttnItem) + 64 * 16 + 8192);
  if (dalloc(h, &h->d_plan, h->plan_cap)) return DEX_ENOMEM;
  if (halloc(h, &h->h_plan, h->plan_cap) || halloc(h, &h->h_best, (R + 2) * 8)) return DEX_ENOMEM;
  // zero-initialised state
  cudaMemsetAsync(h->counters, 0, h->counter_bytes, h->st);
  cudaMemsetAsync(h->attn_counters, 0, h->attn_counter_bytes, h->st);
  cudaMemsetAsync(h->acc64, 0, h->acc_bytes, h->st);
  cudaMemsetAsync(h->err, 0, 16, h->st);
  cudaMemsetAsync(h->kv_commit, 0, B * L * 2 * KVH * ctx * hd * 2, h->st);
  cudaMemsetAsync(h->kv_pool, 0, B * h->n_slots * L * 2 * KVH * hd * 2, h->st);
  cudaMemsetAsync(h->hidden, 0, static_cast<size_t>(h->hrows) * h->d * 4, h->st);
  cudaMemsetAsync(h->hb, 0, 2 * R * h->d * 2, h->st);
  cudaMemsetAsync(h->exit_hb, 0, 2 * R * h->d * 2, h->st);
  cudaMemsetAsync(h->attn_out, 0, 2 * R * qd * 2, h->st);
  cudaMemsetAsync(h->act, 0, 2 * R * h->dff * 2, h->st);
  if (h->ad_act) cudaMemsetAsync(h->ad_act, 0, 2 * R * 2 * static_cast<size_t>(h->d) * 2, h->st);
  // RoPE table (rotate-half, frequencies theta^(-2i/hd)), computed in double
  {
    std::vector<float2> tab(ctx * (hd / 2));
    for (size_t p = 0; p < ctx; ++p)
      for (size_t i = 0; i < hd / 2; ++i) {
        const double inv = pow(static_cast<double>(h->theta), -2.0 * static_cast<double>(i) / static_cast<double>(hd));
        const double ang = static_cast<double>(p) * inv;
        tab[p * (hd / 2) + i] = make_float2(static_cast<float>(cos(ang)), static_cast<float>(sin(ang)));
      }
    if (cudaMemcpy(h->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
      return DEX_ECUDA;
    std::vector<const bf16*> norms(L);
    for (size_t l = 0; l < L; ++l) norms[l] = W(h, static_cast<int>(l), 0);
    if (cudaMemcpy(h->d_attn_norms, norms.data(), L * sizeof(void*), cudaMemcpyHostToDevice) != cudaSuccess)
      return DEX_ECUDA;
  }
  // tensor maps: weights (box 128 rows; gate/up 64 rows) and activation buffers over both
  // planes (2 R rows, box nt rows; the lo box is read plane_rows = R rows below the hi box)
  h->tm_q.resize(L);
  h->tm_k.resize(L);
  h->tm_v.resize(L);
  h->tm_o.resize(L);
  h->tm_g.resize(L);
  h->tm_u.resize(L);
  h->tm_d.resize(L);
  for (size_t l = 0; l < L; ++l) {
    const int li = static_cast<int>(l);
    rc |= encode_2d(&h->tm_q[l], W(h, li, 1), qd, h->d, 128);
    rc |= encode_2d(&h->tm_k[l], W(h, li, 2), kvd, h->d, 128);
    rc |= encode_2d(&h->tm_v[l], W(h, li, 3), kvd, h->d, 128);
    rc |= encode_2d(&h->tm_o[l], W(h, li, 4), h->d, qd, 128);
    rc |= encode_2d(&h->tm_g[l], W(h, li, 6), h->dff, h->d, 64);
    rc |= encode_2d(&h->tm_u[l], W(h, li, 7), h->dff, h->d, 64);
    rc |= encode_2d(&h->tm_d[l], W(h, li, 8), h->d, h->dff, 128);
  }
  rc |= encode_2d(&h->tm_lm, h->lm_head, h->V, h->d, 128);
  // committed K/V rows of hd fp16 elements: [B][L][2][KVH][max_ctx] rows (32-row boxes)
  rc |= encode_2d(&h->tm_kv, h->kv_commit, B * L * 2 * KVH * ctx, hd, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  for (int i = 1; i <= 16; ++i) {
    rc |= encode_2d(&h->tm_hb[i], h->hb, 2 * R, h->d, 16 * i);
    rc |= encode_2d(&h->tm_attn[i], h->attn_out, 2 * R, qd, 16 * i);
    rc |= encode_2d(&h->tm_act[i], h->act, 2 * R, h->dff, 16 * i);
    rc |= encode_2d(&h->tm_exit[i], h->exit_hb, 2 * R, h->d, 16 * i);
    if (h->ad_act) rc |= encode_2d(&h->tm_adact[i], h->ad_act, 2 * R, 2 * h->d, 16 * i);
  }
  if (rc) return DEX_EINVAL;
  // pack every GEMM weight once: contiguous, pre-swizzled 16 KB boxes in streaming order
  {
    const int kb_d = (h->d + 63) / 64, kb_q = (qd + 63) / 64, kb_f = (h->dff + 63) / 64;
    const int t_qkv = (qd + 2 * kvd) / 128, t_o = h->d / 128, t_gu = (h->dff + 63) / 64, t_lm = (h->V + 127) / 128;
    const size_t b_qkv = dex::packed_bytes(t_qkv, kb_d), b_o = dex::packed_bytes(t_o, kb_q);
    const size_t b_gu = dex::packed_bytes(t_gu, kb_d), b_d = dex::packed_bytes(t_o, kb_f);
    const size_t b_lm = dex::packed_bytes(t_lm, kb_d);
    h->packed_total = L * (b_qkv + b_o + b_gu + b_d) + b_lm;
    uint8_t* base = nullptr;
    if (dalloc(h, &base, h->packed_total)) return DEX_ENOMEM;
    using PS = dex::PackSrc;
    const PS none = {nullptr, 0};
    cudaError_t ce = cudaSuccess;
    for (size_t l = 0; l < L; ++l) {
      const int li = static_cast<int>(l);
      uint8_t* pq = base + l * (b_qkv + b_o + b_gu + b_d);
      uint8_t* po = pq + b_qkv;
      uint8_t* pg = po + b_o;
      uint8_t* pd = pg + b_gu;
      h->pk_qkv.push_back(pq);
      h->pk_o.push_back(po);
      h->pk_gu.push_back(pg);
      h->pk_d.push_back(pd);
      if (ce == cudaSuccess)
        ce = dex::launch_pack(dex::PACK_ROWS, PS{W(h, li, 1), qd}, PS{W(h, li, 2), kvd}, PS{W(h, li, 3), kvd}, h->d,
                              t_qkv, pq, h->st);
      if (ce == cudaSuccess)
        ce = dex::launch_pack(dex::PACK_ROWS, PS{W(h, li, 4), h->d}, none, none, qd, t_o, po, h->st);
      if (ce == cudaSuccess)
        ce = dex::launch_pack(dex::PACK_SWIGLU, PS{W(h, li, 6), h->dff}, PS{W(h, li, 7), h->dff}, none, h->d, t_gu,
                              pg, h->st);
      if (ce == cudaSuccess)
        ce = dex::launch_pack(dex::PACK_ROWS, PS{W(h, li, 8), h->d}, none, none, h->dff, t_o, pd, h->st);
    }
    uint8_t* plm = base + L * (b_qkv + b_o + b_gu + b_d);
    h->pk_lm = plm;
    if (ce == cudaSuccess)
      ce = dex::launch_pack(dex::PACK_ROWS, PS{h->lm_head, h->V}, none, none, h->d, t_lm, plm, h->st);
    if (ce != cudaSuccess) return DEX_ECUDA;
    // adapters: W1 [2d][d] (2d/128 tiles over d), W2 [d][2d] (d/128 tiles over 2d)
    if (h->n_adapters) {
      const size_t b_a1 = dex::packed_bytes(2 * h->d / 128, kb_d);
      const size_t b_a2 = dex::packed_bytes(t_o, (2 * h->d + 63) / 64);
      uint8_t* abase = nullptr;
      if (dalloc(h, &abase, h->n_adapters * (b_a1 + b_a2))) return DEX_ENOMEM;
      for (int k = 0; k < h->n_adapters && ce == cudaSuccess; ++k) {
        const void* const* ap = m->adapters + static_cast<size_t>(k) * 5;
        uint8_t* p1 = abase + k * (b_a1 + b_a2);
        uint8_t* p2 = p1 + b_a1;
        h->pk_ad1.push_back(p1);
        h->pk_ad2.push_back(p2);
        ce = dex::launch_pack(dex::PACK_ROWS, PS{static_cast<const bf16*>(ap[1]), 2 * h->d}, none, none, h->d,
                              2 * h->d / 128, p1, h->st);
        if (ce == cudaSuccess)
          ce = dex::launch_pack(dex::PACK_ROWS, PS{static_cast<const bf16*>(ap[3]), h->d}, none, none, 2 * h->d,
                                t_o, p2, h->st);
      }
      if (ce != cudaSuccess) return DEX_ECUDA;
    }
  }
  if (cudaStreamSynchronize(h->st) != cudaSuccess) return DEX_ECUDA;
  *out = hp.release();
  return DEX_OK;
}

int dex_prefill(dex_handle* h, int32_t seq, const int32_t* tokens, int32_t n_tokens) {
  if (!h || !tokens || seq < 0 || seq >= h->cfg.batch || n_tokens < 1) return DEX_EINVAL;
  if (h->broken) return DEX_ECUDA;
  if (n_tokens + h->cfg.max_new + h->N > h->cfg.max_ctx) return DEX_ECAPACITY;
  for (int i = 0; i < n_tokens; ++i)
    if (tokens[i] < 0 || tokens[i] >= h->V) return DEX_EINVAL;
  h->lat->stop(seq);
  h->lat_ar->stop(seq);
  h->mode[seq] = 0;
  h->n_done[seq] = 0;
  auto drop = [&](std::vector<dex_copy_job>& v) {
    v.erase(std::remove_if(v.begin(), v.end(), [&](const dex_copy_job& j) { return j.seq == seq; }), v.end());
  };
  drop(h->pending_jobs);
  drop(h->pending_jobs_ar);
  const int P = n_tokens - 1;   // committed positions 0..P-1 get their KV here
  const int chunk = h->prefill_rows;
  for (int c0 = 0; c0 < P; c0 += chunk) {
    const int n = std::min(chunk, P - c0);
    RoundTables t;
    for (int i = 0; i < n; ++i) {
      dex::DevNode dn = {};
      dn.seq = seq;
      dn.pos = c0 + i;
      dn.c_end = c0 + i + 1;
      dn.slot = 0;
      dn.hrow = h->cfg.batch * h->n_slots + i;
      dn.kv_commit = 1;
      dn.token = tokens[c0 + i];
      dn.first_layer = 0;
      dn.unmasked = 1;
      t.nodes.push_back(dn);
    }
    // GEMM groups of prefill_group_rows rows (the same layer's weights, read once from HBM
    // and by the later groups from L2), attention items of one MMA pass each (rows x query
    // heads per KV head <= 16): the (item, KV head) combinations spread over the grid, and
    // early rows skip late key groups
    const int rows_per_item = std::max(1, dex::kAttnPassQueries / (h->H / h->KVH));
    std::vector<Batch> batches;
    for (int g0 = 0; g0 < n; g0 += h->prefill_group_rows) {
      Batch b;
      b.off = g0;
      b.n = std::min(h->prefill_group_rows, n - g0);
      b.l0 = 0;
      b.l1 = h->L;
      for (int r0 = g0; r0 < g0 + b.n; r0 += rows_per_item) {
        dex::AttnItem it = {};
        it.seq = seq;
        it.row_begin = r0;
        it.row_end = std::min(g0 + b.n, r0 + rows_per_item);
        it.max_pos = c0 + it.row_end - 1;
        it.max_cend = c0 + it.row_end;
        it.n_groups = std::max(1, (dex::attn_bulk_end(it.max_pos) + dex::kAttnGroupPos - 1) / dex::kAttnGroupPos);
        b.items.push_back(it);
      }
      batches.push_back(std::move(b));
    }
    const std::vector<Slot> slots = build_slots(batches, h->KVH, &t);
    Uploaded u;
    int rc = upload(h, t, &u);
    if (rc) return rc;
    dex::AssembleArgs aa = {};
    aa.nodes = u.nodes;
    aa.n_rows = n;
    aa.d = h->d;
    aa.embed = h->embed;
    aa.attn_norm = h->d_attn_norms;
    aa.hidden = h->hidden;
    aa.hb = h->hb;
    aa.plane_rows = h->rows_cap;
    aa.ssq = h->ssq;
    aa.best = nullptr;
    cudaError_t ce = dex::launch_assemble(aa, h->st, false);
    if (ce != cudaSuccess) return cuda_fail(h, ce);
    rc = run_layers(h, u, batches, slots, false, true);
    if (rc) return rc;
    // the upload buffer is reused by the next chunk: wait for this chunk
    if (cudaMemcpyAsync(h->h_best, h->err, 4, cudaMemcpyDeviceToHost, h->st) != cudaSuccess ||
        cudaStreamSynchronize(h->st) != cudaSuccess)
      return cuda_fail(h, cudaGetLastError());
    const int32_t dev_err = static_cast<int32_t>(h->h_best[0] & 0xffffffffull);
    if (dev_err) return check_device_error(h, dev_err);
    // per-launch timings cover decode rounds only: drop the prefill's events
    h->gemm_events.clear();
    h->attn_events.clear();
    h->ev_used = 0;
  }
  h->lat->start(seq, n_tokens, tokens[n_tokens - 1]);
  h->lat_ar->start(seq, n_tokens, tokens[n_tokens - 1]);
  return DEX_OK;
}

static int step_common(dex_handle* h, bool ar, int32_t* out_tokens, int32_t* n_committed) {
  if (!h || !out_tokens || !n_committed) return DEX_EINVAL;
  dex::Lattice* lat = ar ? h->lat_ar.get() : h->lat.get();
  dex::Lattice* other = ar ? h->lat.get() : h->lat_ar.get();
  const int want = ar ? 2 : 1;
  for (int b = 0; b < h->cfg.batch; ++b) {
    if (!lat->active(b)) continue;
    if (h->mode[b] != 0 && h->mode[b] != want) return DEX_ESTATE;
  }
  for (int b = 0; b < h->cfg.batch; ++b)
    if (lat->active(b)) {
      h->mode[b] = want;
      other->stop(b);
    }
  return run_round(h, lat, ar ? &h->pending_jobs_ar : &h->pending_jobs, out_tokens, n_committed);
}

int dex_step(dex_handle* h, int32_t* out_tokens, int32_t* n_committed) {
  return step_common(h, false, out_tokens, n_committed);
}
int dex_ar_step(dex_handle* h, int32_t* out_tokens, int32_t* n_committed) {
  return step_common(h, true, out_tokens, n_committed);
}

static int generate_loop(dex_handle* h, bool ar, int32_t* out) {
  if (!h || !out) return DEX_EINVAL;
  std::vector<int32_t> tok(h->cfg.batch), nc(h->cfg.batch);
  dex::Lattice* lat = ar ? h->lat_ar.get() : h->lat.get();
  while (lat->any_active()) {
    const int rc = step_common(h, ar, tok.data(), nc.data());
    if (rc) return rc;
    for (int b = 0; b < h->cfg.batch; ++b)
      if (nc[b]) out[static_cast<size_t>(b) * h->cfg.max_new + h->n_done[b] - 1] = tok[b];
  }
  return DEX_OK;
}

int dex_generate(dex_handle* h, int32_t* out) { return generate_loop(h, false, out); }
int dex_ar_generate(dex_handle* h, int32_t* out) { return generate_loop(h, true, out); }

int dex_get_stats(const dex_handle* h, dex_stats* out) {
  if (!h || !out) return DEX_EINVAL;
  *out = h->stats;
  return DEX_OK;
}
int dex_reset_stats(dex_handle* h) {
  if (!h) return DEX_EINVAL;
  h->stats = dex_stats{};
  h->gemm_events.clear();
  h->attn_events.clear();
  return DEX_OK;
}
int dex_set_timing(dex_handle* h, int32_t level) {
  if (!h || level < 0 || level > 3) return DEX_EINVAL;
  if (level == 3 && !h->timeline && getenv("DEX_TIMELINE")) {
    const char* n = getenv("DEX_TIMELINE_LAUNCHES");
    h->tl_cap = n ? std::max(1, atoi(n)) : 512;
    const size_t bytes = static_cast<size_t>(h->tl_cap) * h->gemm_ctas * dex::kTimelineSlots * 8;
    if (dalloc(h, &h->timeline, bytes) || cudaMemset(h->timeline, 0, bytes) != cudaSuccess) return DEX_ENOMEM;
    h->atl_cap = h->tl_cap;
    const size_t abytes = static_cast<size_t>(h->atl_cap) * h->n_sm * dex::kAttnTimelineSlots * 8;
    if (dalloc(h, &h->atl, abytes) || cudaMemset(h->atl, 0, abytes) != cudaSuccess) return DEX_ENOMEM;
  }
  h->timing = level;
  return DEX_OK;
}

int dex_last_round_nodes(const dex_handle* h, int32_t* host_out, int32_t max_rows, int32_t* rows_out) {
  if (!h || !rows_out) return DEX_EINVAL;
  const int n = static_cast<int>(h->last_plan.size());
  *rows_out = n;
  if (n > max_rows || (n && !host_out)) return DEX_ECAPACITY;
  for (int k = 0; k < n; ++k) {
    const auto& p = h->last_plan[k];
    int32_t* o = host_out + 8 * k;
    o[0] = p.seq;
    o[1] = p.heap;
    o[2] = p.stage;
    o[3] = p.plen;
    o[4] = p.target_pos;
    o[5] = h->last_tokens[k];
    o[6] = p.n_prior;
    o[7] = p.pos;
  }
  return DEX_OK;
}

int dex_debug_logits(dex_handle* h, float* host_out, int32_t max_rows, int32_t* rows_out) {
  if (!h || !rows_out) return DEX_EINVAL;
  if (!h->cfg.debug_logits) return DEX_ESTATE;
  const int n = static_cast<int>(h->last_plan.size());
  *rows_out = n;
  if (n > max_rows || (n && !host_out)) return DEX_ECAPACITY;
  if (cudaMemcpyAsync(host_out, h->logits_dbg, static_cast<size_t>(n) * h->V * 4, cudaMemcpyDeviceToHost, h->st) !=
          cudaSuccess ||
      cudaStreamSynchronize(h->st) != cudaSuccess)
    return cuda_fail(h, cudaGetLastError());
  return DEX_OK;
}

// ---- failure-path self-test --------------------------------------------------------------

// The bounded mbarrier wait every pipeline of the library uses, against a barrier that
// nothing arrives on: it gives up after limit_ns and raises the device error flag exactly
// as a stalled GEMM or attention pipeline would.  No copy or MMA is issued against the
// barrier, so nothing is in flight when the kernel returns.
__global__ void stall_probe_kernel(int32_t* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    dex::mbar_init(&bar, 1);
    dex::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) dex::mbar_wait(&bar, 0, err, dex::DEV_TIMEOUT_FULL, limit_ns);
}

int dex_selftest_stall(dex_handle* h, int32_t limit_us) {
  if (!h || limit_us < 1 || limit_us > 1000000) return DEX_EINVAL;
  if (h->broken) return DEX_ECUDA;
  const unsigned long long limit_ns = static_cast<unsigned long long>(limit_us) * 1000ull;
  int32_t* err = h->err;
  void* args[] = {&err, const_cast<unsigned long long*>(&limit_ns)};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = h->st;
  if (cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(stall_probe_kernel), args) != cudaSuccess)
    return cuda_fail(h, cudaGetLastError());
  // the same read-back and check as the end of a decode round
  if (cudaMemcpyAsync(h->h_best, h->err, sizeof(int32_t), cudaMemcpyDeviceToHost, h->st) !=
          cudaSuccess ||
      cudaStreamSynchronize(h->st) != cudaSuccess)
    return cuda_fail(h, cudaGetLastError());
  const int32_t flag = static_cast<int32_t>(h->h_best[0] & 0xffffffffull);
  return check_device_error(h, flag);
}

// ---- kernels in isolation ---------------------------------------------------------------

static_assert(sizeof(dex_exit_node) == 5 * sizeof(int32_t), "dex_exit_node is five int32 fields");

int dex_exit_head_decs(const void* hidden, int32_t n, int32_t d, const void* final_norm, float rms_eps,
                       const void* lm_head, int32_t vocab, const dex_exit_node* nodes, const int32_t* priors,
                       int32_t sample, float tau, uint64_t seed, int32_t* tokens, float* logits, void* stream) {
  if (!hidden || !final_norm || !lm_head || !nodes || !tokens || n < 1 || n > 256 || d < 128 || d % 128 || d > 8192 ||
      vocab < 2 || (sample && !(tau > 0)))
    return DEX_EINVAL;
  if (get_encoder()) return DEX_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DEX_ENODEV;
  const int n_tiles = (vocab + 127) / 128, kb = (d + 63) / 64;
  const int nt = (n + 15) & ~15;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t o_hb = 0, o_ssq = o_hb + up(static_cast<size_t>(2) * nt * d * 2);   // hi/lo planes of nt rows
  const size_t o_best = o_ssq + up(static_cast<size_t>(n) * (d / 128) * 4);
  const size_t o_nodes = o_best + up(static_cast<size_t>(n) * 8);
  const size_t o_cnt = o_nodes + up(static_cast<size_t>(n) * sizeof(dex::DevNode));
  const size_t o_err = o_cnt + up(static_cast<size_t>(n_tiles) * 4);
  const size_t o_part = o_err + 256;
  const int ctas = 2 * n_sm;   // two CTAs per SM, as in the decoder (104 KB shared memory each)
  const int segs = dex::gemm_segments(n_tiles, kb, ctas);
  const size_t total = o_part + (segs > 1 ? dex::gemm_partial_bytes(nt, static_cast<size_t>(n_tiles) * segs) : 256);
  uint8_t* scratch = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&scratch), total, st) != cudaSuccess) return DEX_ENOMEM;
  bf16* hb = reinterpret_cast<bf16*>(scratch + o_hb);
  float* ssq = reinterpret_cast<float*>(scratch + o_ssq);
  unsigned long long* best = reinterpret_cast<unsigned long long*>(scratch + o_best);
  dex::DevNode* dn = reinterpret_cast<dex::DevNode*>(scratch + o_nodes);
  int32_t* cnt = reinterpret_cast<int32_t*>(scratch + o_cnt);
  int rc = DEX_OK;
  CUtensorMap tm_w, tm_b;
  if (encode_2d(&tm_w, lm_head, vocab, d, 128) || encode_2d(&tm_b, hb, 2 * nt, d, nt)) rc = DEX_EINVAL;
  if (!rc) {
    cudaMemsetAsync(hb, 0, static_cast<size_t>(2) * nt * d * 2, st);
    cudaMemsetAsync(cnt, 0, o_part - o_cnt, st);   // arrival counters and the error flag
    if (dex::launch_exit_prep(static_cast<const bf16*>(hidden), n, d, static_cast<const bf16*>(final_norm), hb, nt, ssq,
                              best, st) != cudaSuccess)
      rc = DEX_ECUDA;
    if (!rc && dex::launch_exit_nodes(nodes, n, dn, st) != cudaSuccess) rc = DEX_ECUDA;
    dex::GemmArgs a = {};
    a.n_groups = 1;
    a.n_ctas = ctas;
    a.n_segs = segs;
    a.groups[0].n = n;
    a.groups[0].b_row0 = 0;
    a.nt = nt;
    a.kblocks = kb;
    a.stages = dex::gemm_stages_for(nt, dex::EPI_EXIT);
    a.n_tiles = n_tiles;
    a.src_tiles0 = n_tiles;
    a.tmem_cols = pow2_at_least(nt);
    a.partial = reinterpret_cast<float*>(scratch + o_part);
    a.counters = cnt;
    a.err = reinterpret_cast<int32_t*>(scratch + o_err);
    a.nodes = dn;
    a.evict_first = 1;
    a.plane_rows = nt;
    a.d = d;
    a.vocab = vocab;
    a.eps = rms_eps;
    a.ssq_in = ssq;
    a.logits_dbg = logits;
    a.best = best;
    a.priors = priors;
    a.sample = sample;
    a.tau = tau;
    a.seed = seed;
    if (!rc && dex::launch_gemm(dex::EPI_EXIT, tm_w, tm_w, tm_w, tm_b, a, st, false) != cudaSuccess) rc = DEX_ECUDA;
    if (!rc && dex::launch_decode_best(best, n, a.err, tokens, st) != cudaSuccess) rc = DEX_ECUDA;
  }
  cudaFreeAsync(scratch, st);
  return rc;
}

int dex_kv_collapse(void* committed, const void* pool, const dex_kv_geom* g, const dex_copy_job* jobs, int32_t n_jobs,
                    int32_t* rejected, void* stream) {
  if (!committed || !pool || !g || (!jobs && n_jobs) || n_jobs < 0 || n_jobs > 65535 || g->head_dim < 8 ||
      g->head_dim % 8 || g->batch < 1 || g->n_layers < 1 || g->n_kv_heads < 1 || g->max_ctx < 1 || g->n_slots < 1)
    return DEX_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rejected && cudaMemsetAsync(rejected, 0, sizeof(int32_t), st) != cudaSuccess) return DEX_ECUDA;
  dex::CollapseArgs a = {};
  a.jobs = reinterpret_cast<const dex::CopyJob*>(jobs);
  a.n_jobs = n_jobs;
  a.kv_commit = committed;
  a.kv_pool = pool;
  a.batch = g->batch;
  a.L = g->n_layers;
  a.KVH = g->n_kv_heads;
  a.row_bytes = g->head_dim * 2;   // bf16 caches
  a.max_ctx = g->max_ctx;
  a.n_slots = g->n_slots;
  a.rejected = rejected;
  const cudaError_t e = dex::launch_collapse(a, st, false);
  if (e == cudaErrorInvalidValue) return DEX_EINVAL;
  return e == cudaSuccess ? DEX_OK : DEX_ECUDA;
}

}  // extern "C"

// ---- exit head + DECS without any allocation ------------------------------------------------
//
// For callers that cannot allocate device memory while they run: code executing inside a
// region that is being captured into a CUDA graph on a stream whose allocator they do not
// own, embedders whose memory budget is fixed up front, or real-time loops that must not
// hit the driver's allocator.  The scratch of dex_exit_head_decs lives instead in one
// file-scope device array, present on every GPU that loads this library until the process
// exits.  Its device address is looked up once per device, on that device's first call.

static __device__ __align__(256) unsigned char g_exit_scratch[DEX_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_exit_scratch_mu;
void* g_exit_scratch_addr[256] = {};   // device ordinal -> address of g_exit_scratch there

// The array's name is only a host-side handle; the kernels need its device address,
// which cudaGetSymbolAddress returns for the device that is current.
int exit_scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= 256) return DEX_ENODEV;
  std::lock_guard<std::mutex> lock(g_exit_scratch_mu);
  if (!g_exit_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_exit_scratch) != cudaSuccess || !p) return DEX_ECUDA;
    g_exit_scratch_addr[dev] = p;
  }
  *out = g_exit_scratch_addr[dev];
  return DEX_OK;
}
}  // namespace

extern "C" int dex_exit_head_decs_noalloc(const void* hidden, int32_t n, int32_t d, const void* final_norm,
                                          float rms_eps, const void* lm_head, int32_t vocab,
                                          const dex_exit_node* nodes, const int32_t* priors, int32_t sample,
                                          float tau, uint64_t seed, int32_t* tokens, float* logits, void* stream) {
  if (!hidden || !final_norm || !lm_head || !nodes || !tokens || n < 1 || n > 256 || d < 128 || d % 128 || d > 8192 ||
      vocab < 2 || (sample && !(tau > 0)))
    return DEX_EINVAL;
  if (get_encoder()) return DEX_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DEX_ENODEV;
  // same scratch layout as dex_exit_head_decs
  const int n_tiles = (vocab + 127) / 128, kb = (d + 63) / 64;
  const int nt = (n + 15) & ~15;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t o_hb = 0, o_ssq = o_hb + up(static_cast<size_t>(2) * nt * d * 2);   // hi/lo planes of nt rows
  const size_t o_best = o_ssq + up(static_cast<size_t>(n) * (d / 128) * 4);
  const size_t o_nodes = o_best + up(static_cast<size_t>(n) * 8);
  const size_t o_cnt = o_nodes + up(static_cast<size_t>(n) * sizeof(dex::DevNode));
  const size_t o_err = o_cnt + up(static_cast<size_t>(n_tiles) * 4);
  const size_t o_part = o_err + 256;
  const int segs = dex::gemm_segments(n_tiles, kb, n_sm);
  const size_t total = o_part + (segs > 1 ? dex::gemm_partial_bytes(nt, static_cast<size_t>(n_tiles) * segs) : 256);
  if (total > DEX_NOALLOC_SCRATCH_BYTES) return DEX_ECAPACITY;   // does not fit the fixed scratch
  void* base = nullptr;
  const int rc0 = exit_scratch_address(dev, &base);
  if (rc0) return rc0;
  uint8_t* scratch = static_cast<uint8_t*>(base);
  bf16* hb = reinterpret_cast<bf16*>(scratch + o_hb);
  float* ssq = reinterpret_cast<float*>(scratch + o_ssq);
  unsigned long long* best = reinterpret_cast<unsigned long long*>(scratch + o_best);
  dex::DevNode* dn = reinterpret_cast<dex::DevNode*>(scratch + o_nodes);
  int32_t* cnt = reinterpret_cast<int32_t*>(scratch + o_cnt);
  CUtensorMap tm_w, tm_b;
  if (encode_2d(&tm_w, lm_head, vocab, d, 128) || encode_2d(&tm_b, hb, 2 * nt, d, nt)) return DEX_EINVAL;
  // the array keeps the previous call's contents: clear what the kernels expect at zero
  // (padding rows of the node tile, split-K arrival counters, the stall flag)
  if (cudaMemsetAsync(hb, 0, static_cast<size_t>(2) * nt * d * 2, st) != cudaSuccess ||
      cudaMemsetAsync(cnt, 0, o_part - o_cnt, st) != cudaSuccess)
    return DEX_ECUDA;
  if (dex::launch_exit_prep(static_cast<const bf16*>(hidden), n, d, static_cast<const bf16*>(final_norm), hb, nt, ssq,
                            best, st) != cudaSuccess)
    return DEX_ECUDA;
  if (dex::launch_exit_nodes(nodes, n, dn, st) != cudaSuccess) return DEX_ECUDA;
  dex::GemmArgs a = {};
  a.n_groups = 1;
  a.n_ctas = n_sm;
  a.n_segs = segs;
  a.groups[0].n = n;
  a.groups[0].b_row0 = 0;
  a.nt = nt;
  a.kblocks = kb;
  a.stages = dex::gemm_stages_for(nt, dex::EPI_EXIT, 200 * 1024);   // one CTA per SM: a deeper ring
  a.n_tiles = n_tiles;
  a.src_tiles0 = n_tiles;
  a.tmem_cols = pow2_at_least(nt);
  a.partial = reinterpret_cast<float*>(scratch + o_part);
  a.counters = cnt;
  a.err = reinterpret_cast<int32_t*>(scratch + o_err);
  a.nodes = dn;
  a.evict_first = 1;
  a.plane_rows = nt;
  a.d = d;
  a.vocab = vocab;
  a.eps = rms_eps;
  a.ssq_in = ssq;
  a.logits_dbg = logits;
  a.best = best;
  a.priors = priors;
  a.sample = sample;
  a.tau = tau;
  a.seed = seed;
  if (dex::launch_gemm(dex::EPI_EXIT, tm_w, tm_w, tm_w, tm_b, a, st, false) != cudaSuccess) return DEX_ECUDA;
  if (dex::launch_decode_best(best, n, a.err, tokens, st) != cudaSuccess) return DEX_ECUDA;
  return DEX_OK;
}

// Shared host/device definitions: the per-node round descriptor, kernel argument
// blocks and the launchers of the DEX kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dex {

// Error flags written by kernels (read back by the host after each round).
enum DevErr : int { DEV_OK = 0, DEV_TIMEOUT_FULL = 1, DEV_TIMEOUT_EMPTY = 2, DEV_TIMEOUT_ACC = 3,
                    DEV_BAD_INDEX = 4, DEV_RANGE = 5 };

// One lattice node of the current round, as the kernels see it.  Node rows are ordered
// by stage; the rows of stage s form one contiguous batch for that stage's layers, and
// the same row index addresses the node in every activation buffer and in the exit head.
struct DevNode {
  int32_t seq;         // sequence
  int32_t pos;         // absolute position of the input token
  int32_t c_end;       // keys at positions < c_end live in the committed cache
  int32_t slot;        // pool slot of the slot chain (branch KV)
  int32_t hrow;        // row of the fp32 hidden-state array (slot chain or prefill scratch)
  int32_t kv_commit;   // 1: this node's K/V are written to the committed cache at pos
  int32_t token;       // stage-0 input token (embedding row), -1 for depth children
  int32_t first_layer; // first layer (0-based) of the node's stage
  int32_t tail_off;    // tail slots (positions c_end..pos) start here in the tail array
  int32_t n_tail;
  int32_t target_pos;  // position being predicted (Gumbel row key)
  int32_t unmasked;    // 1: final-depth reference, no DECS mask
  int32_t prior_off;   // DECS prior tokens start here in the prior array
  int32_t n_prior;
  int32_t pad0, pad1;
};
static_assert(sizeof(DevNode) == 64, "DevNode is 64 bytes");

// Key positions per attention CTA (four 32-key warp slices); groups are aligned to position 0.
constexpr int kAttnGroupPos = 128;
constexpr int kAttnMaxGroups = 32;   // max_ctx <= 4096
constexpr int kAttnPassQueries = 16; // queries of one attention pass (the MMA's N)
// A query at position p takes keys [max(0, p - kAttnWindow + 1), p] on CUDA cores and the
// older ones on the tensor cores; the window exceeds every node's branch depth (|X| <= 10),
// so the tensor-core keys are always committed ones.
constexpr int kAttnWindow = 16;
inline int attn_bulk_end(int pos) { return pos - kAttnWindow + 1 > 0 ? pos - kAttnWindow + 1 : 0; }

// Attention work item: one sequence's contiguous node rows within a stage batch.
struct AttnItem {
  int32_t seq, row_begin, row_end;   // absolute node rows
  int32_t max_pos, max_cend;         // largest input position / committed extent among the rows
  int32_t n_groups;                  // kAttnGroupPos-position key groups covering the bulk keys (>= 1)
  int32_t counter;                   // index of this item's merge counters (x KVH)
  int32_t layer;                     // decoder layer of this item (items of several stages share a launch)
  int32_t unit0;                     // first (item, KV head, group) unit of the item in its launch
  int32_t pad0;
};

// EPI_ADUP / EPI_ADDOWN: the two layers of an inducing adapter at a non-final exit.
enum SumMode : int { SUM_FP32 = 0, SUM_FIXED_RED = 2 };
enum Epi : int { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_EXIT = 3, EPI_ADUP = 4, EPI_ADDOWN = 5 };

// One weight matrix of a grouped launch: a stage's layer and that stage's node rows.  The
// groups of a launch share the weight shape; each keeps its own fixed work partition.
constexpr int kMaxGroups = 10;
struct GemmGroup {
  const uint8_t* a_packed;    // packed weights of this group's layer (null: TMA from tmA*)
  const __nv_bfloat16* g_next;// RESID: gain of the next norm (null at the model's end)
  const __nv_bfloat16* g_exit;// RESID at a stage end: gain of the exit input (null: g_final;
                              // an adapter's RMSNorm gain when the stage's exit is adapted)
  const __nv_bfloat16* bias;  // ADUP: b1, ADDOWN: b2
  int32_t b_row0;       // first node row (= first B row)
  int32_t n;            // node rows
  int32_t layer;        // decoder layer (QKV: KV cache addressing)
  int32_t stage_end;    // RESID: last layer of the stage -> also write the exit-head input
  int32_t has_next;     // RESID: write the next layer's bf16 input
  float alpha;          // ADDOWN: the adapter's scalar gate
};

struct GemmArgs {
  // tiling
  int32_t n_groups;     // weight matrices in this launch
  int32_t n_ctas;       // grid size (resident CTAs); units are dealt out over it
  int32_t n_segs;       // k segments per output tile (fixed per weight shape)
  int32_t nt;           // node tile (multiple of 16, <= 256) >= every group's n
  int32_t kblocks;      // K / 64, rounded up
  int32_t stages;       // smem pipeline depth
  int32_t n_tiles;      // output tiles
  int32_t src_tiles0, src_tiles1;   // tiles of source 0 and 1 (source 2 takes the rest)
  int32_t tmem_cols;
  float* partial;       // [n_groups][n_tiles][n_segs][128][nt] fp32 segment partials
  // How a tile's k segments are summed: SUM_FP32 -- fp32 partial tiles added in segment
  // order; SUM_FIXED_RED (decoder-layer epilogues) -- each segment adds its
  // partial at L2 (red.add) into acc in 2^-32 fixed point, where the sum is exact.  A
  // decoder uses one of the two for every layer launch, so results do not depend on the batch.
  int32_t sum_mode;
  long long* acc;       // SUM_FIXED_RED: [n_groups][n_tiles][nt][128] int64, zero at rest
  int32_t* counters;    // [n_groups][n_tiles] arrival counters (left at 0)
  int32_t* err;         // device error flag
  const DevNode* nodes; // node rows (absolute)
  int32_t evict_first;  // stream A with an L2 evict-first policy
  // Activation buffers hold two bf16 planes, hi then lo (x ~= hi + lo): the lo plane of a
  // [rows][K] buffer starts plane_rows rows after the hi plane, for the B operand (tensor
  // map over 2 * plane_rows rows) and for every activation the epilogue writes.
  int32_t plane_rows;
  // model geometry
  int32_t d, H, KVH, hd, L, d_ff, vocab, max_ctx, n_slots;
  float eps;
  // RMSNorm inputs (QKV, SWIGLU, EXIT): per-row 128-feature partial sums of squares
  const float* ssq_in;  // [rows][d/128]
  // QKV
  float* q_out;         // [rows][H*hd]
  __half* kv_commit;    // [B][L][2][KVH][max_ctx][hd] fp16
  __half* kv_pool;      // [B][n_slots][L][2][KVH][hd] fp16
  const float2* rope;   // [max_ctx][hd/2] (cos, sin)
  // RESID
  float* hidden;        // [hrows][d]
  __nv_bfloat16* hb_out;      // [2][rows][d]  pair of h * g_next, next layer's input
  float* ssq_out;       // [rows][d/128]
  __nv_bfloat16* exit_hb;     // [2][rows][d]  pair of h * g_final
  const __nv_bfloat16* g_final;
  float* exit_ssq;      // [rows][d/128]
  // SWIGLU (and ADUP: [2][rows][2d], d_ff = 2d)
  __nv_bfloat16* act_out;     // [2][rows][d_ff]  pair of SiLU(gate) * up
  // EXIT + DECS
  float* logits_dbg;    // [rows][vocab] or null
  unsigned long long* best;   // [rows] packed (score, ~token), zeroed before the launch
  const int32_t* priors;
  int32_t sample;
  float tau;
  unsigned long long seed;
  // diagnostics: per-CTA records of kTimelineSlots words, or null (see gemm.cu)
  unsigned long long* timeline;
  GemmGroup groups[kMaxGroups];
};
constexpr int kTimelineUnits = 48;
constexpr int kTimelineSlots = 4 + 3 * kTimelineUnits;

// The committed cache is read through a TMA tensor map (fp16 rows of hd elements, box
// 64 x 32 rows, 128-byte swizzle); the branch pool through kv_pool.
struct AttnArgs {
  const DevNode* nodes;
  const AttnItem* items;
  int32_t n_items, n_units;    // items of the launch; units = sum over items of KVH x n_groups
  const int32_t* tails;
  const float* q;              // [rows][H*hd]
  const __half* kv_commit;     // fp16 committed cache (window keys; layout as in GemmArgs)
  const __half* kv_pool;       // fp16 pool (layout as in GemmArgs)
  __nv_bfloat16* out;          // [2][plane_rows][H*hd] hi/lo pair
  int32_t plane_rows;
  float* part;                 // [rows][H][part_slots][hd + 2]: group records, then the window record
  int32_t* counters;           // [items * KVH]
  int32_t* err;
  int32_t H, KVH, hd, L, max_ctx, n_slots, part_slots;   // part_slots = key groups of max_ctx + 1
  float scale_log2;            // log2(e) / sqrt(hd)
  // 1: every bulk key was committed before the launch's predecessor ran (a decode round:
  // bulk keys precede the round's committed extent, and rounds are host-synchronised), so
  // the K/V producer streams them without waiting for that kernel; 0 (prefill): it waits
  int32_t early_kv;
  // diagnostics: per-CTA records of kAttnTimelineSlots words (globaltimer ns), or null:
  // [0] epilogue start, [1] epilogue end, [2] units, then per unit (first kAttnTimelineUnits)
  // query tile posted, scores seen, scores reduced, maxima shared, probabilities posted,
  // output seen, partials written, unit counted; then up to four combinations (start, end)
  unsigned long long* timeline;
};
// Causal attention of one prefill pass: the pass's node rows are consecutive prompt
// positions of one sequence whose K/V (every position up to the row's own) are in the
// committed cache.  One CTA per (block of 128 query rows, KV head): rows are position-major,
// 128 / G positions x the G query heads of the KV head.
struct PrefillAttnArgs {
  const DevNode* nodes;        // the pass's node rows 0 .. n_rows-1 (positions in .pos)
  int32_t n_rows, seq, layer;
  const float* q;              // [rows][H*hd]
  __nv_bfloat16* out;          // [2][plane_rows][H*hd] hi/lo pair
  int32_t plane_rows;
  int32_t* err;
  int32_t H, KVH, hd, L, max_ctx;
  float scale_log2;            // log2(e) / sqrt(hd)
};
constexpr int kAttnTimelineUnits = 12;
constexpr int kAttnTimelineSlots = 3 + 8 * kAttnTimelineUnits + 8;

struct AssembleArgs {
  const DevNode* nodes;
  int32_t n_rows;
  int32_t d;
  const __nv_bfloat16* embed;          // [V][d]
  const __nv_bfloat16* const* attn_norm;  // device array [L] of gains
  float* hidden;
  __nv_bfloat16* hb;                    // [2][plane_rows][d] hi/lo pair
  int32_t plane_rows;
  float* ssq;
  unsigned long long* best;             // zeroed for rows 0..n_rows-1 (may be null)
};

struct CopyJob { int32_t seq, slot, pos, n_layers; };

// KV rows are copied as raw bytes: row_bytes = head_dim x element size (fp16 caches of the
// decoder, bf16 caches of the isolated entry point), a multiple of 16.
// A job whose sequence, slot, position or layer count is out of range is skipped (nothing
// is read or written for it): it sets *err to DEV_BAD_INDEX and adds one to *rejected
// (either may be null).
struct CollapseArgs {
  const CopyJob* jobs;
  int32_t n_jobs;
  void* kv_commit;
  const void* kv_pool;
  int32_t batch, L, KVH, row_bytes, max_ctx, n_slots;
  int32_t* err;
  int32_t* rejected;
};

// ---- launchers (return cudaError_t of the launch) -----------------------------------------
// A tensor maps: up to three weight sources (QKV: wq, wk, wv; SWIGLU: wg, wu with 64-row
// boxes); B: the activation rows with a box of nt rows.
// Persistent launch over n_ctas CTAs: the launch's (group, tile, k-segment) units are cut
// into one contiguous range per CTA; stages chosen from the node tile.
cudaError_t launch_gemm(int epi, const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& a2,
                        const CUtensorMap& b, const GemmArgs& args, cudaStream_t st, bool pdl);
size_t gemm_smem_bytes(int nt, int stages, int epi);
// Ring depth for node tile nt and epilogue epi: the most stages (2..8) that fit the budget
// (small node tiles) or the opt-in limit (the wide tiles of prefill).
int gemm_stages_for(int nt, int epi, size_t small_budget = 104 * 1024);
// k segments per 128-row tile for a weight of n_tiles tiles and kblocks k-blocks on a grid
// of n_ctas CTAs (depends on nothing else, so results never depend on the batch).
int gemm_segments(int n_tiles, int kblocks, int n_ctas);
// Bytes of the segment-partial workspace of a launch with `units` (group, tile, segment)
// units and node tile nt (none is needed when every tile has one segment).
inline size_t gemm_partial_bytes(int nt, size_t units) { return units * nt * 128 * 4; }
// max_nq: the largest number of queries (node rows x query heads per KV head) of an item.
// Preferred shared-memory carveout (percent) applied to every kernel of the library, or -1
// for the driver's choice: DEX_SMEM_CARVEOUT, read once (diagnostics / tuning).
int smem_carveout_pref();
template <typename F>
inline cudaError_t apply_carveout(F* func) {
  const int c = smem_carveout_pref();
  if (c < 0) return cudaSuccess;
  return cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, c);
}

// Persistent launch over min(n_units, n_ctas) CTAs (one per SM); items with more than
// kAttnPassQueries queries take several passes.
cudaError_t launch_attention(const CUtensorMap& tm_kv, const AttnArgs& a, int n_ctas, cudaStream_t st, bool pdl);
// false when the shape has no prefill kernel (head_dim not 64/128, or 128 not a multiple of
// the query heads per KV head): prefill passes then use launch_attention.
bool prefill_attention_supported(int H, int KVH, int hd);
cudaError_t launch_prefill_attention(const CUtensorMap& tm_kv, const PrefillAttnArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_assemble(const AssembleArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_collapse(const CollapseArgs& a, cudaStream_t st, bool pdl);
// bf16 [n][d] rows -> hi/lo pair of h * g ([2][plane_rows][d]) and partial sums of squares
// (the exit-head input of an isolated exit-head call); zeroes the argmax slots.
cudaError_t launch_exit_prep(const __nv_bfloat16* h, int n, int d, const __nv_bfloat16* g,
                             __nv_bfloat16* hb, int plane_rows, float* ssq, unsigned long long* best,
                             cudaStream_t st);
// Packed GEMM weights: box (t, k) = rows 128t..128t+127 x columns 64k..64k+63 of the
// (virtual) weight matrix, stored at byte offset (t * kblocks + k) * 16384 in the 128-byte
// swizzled K-major shared-memory image (chunk c of row r at r*128 + (c ^ (r & 7))*16).
// Modes: PACK_ROWS stacks up to three row-major sources (QKV: wq, wk, wv); PACK_SWIGLU
// puts 64 rows of src0 (gate) over the same 64 rows of src1 (up) in each tile.  Rows and
// columns outside the sources are zero.
enum PackMode : int { PACK_ROWS = 0, PACK_SWIGLU = 1 };
struct PackSrc { const __nv_bfloat16* ptr; int32_t rows; };
size_t packed_bytes(int n_tiles, int kblocks);
cudaError_t launch_pack(int mode, PackSrc s0, PackSrc s1, PackSrc s2, int K, int n_tiles, uint8_t* out,
                        cudaStream_t st);
// tokens[i] = the token packed in best[i]; every token is -1 when *err is set (a bounded
// wait of the exit-head GEMM gave up, so the argmax slots are incomplete).
cudaError_t launch_decode_best(const unsigned long long* best, int n, const int32_t* err, int32_t* tokens,
                               cudaStream_t st);
// Node table of an isolated exit-head call (host struct dex_exit_node, device array) ->
// the kernels' DevNode rows.
cudaError_t launch_exit_nodes(const void* exit_nodes, int n, DevNode* out, cudaStream_t st);

}  // namespace dex

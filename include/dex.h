/*
 * dex.h -- C ABI of the GB300 (sm_103a) Depth Exploration Decoding library.
 *
 * Depth Exploration Decoding (DEX), "Depth Exploration for LLM Decoding"
 * (arXiv 2606.29223): each expand-commit-collapse cycle expands a depth-position
 * lattice of exploration tokens (section 3.2, Figure 2), decodes every node with
 * depth-coupled sampling (section 3.3, Appendix C.1 Algorithm 2), commits the
 * final-depth token y = u_{N-1}, keeps the shallowest anchor branch with u_k = y and
 * collapses the lattice onto it (Algorithm 1, expand / DECS / insert /
 * validate_and_commit / collapse / advance).
 *
 * On one GPU, a round batches every live lattice node of every sequence into one
 * pass: the decoder-layer slice (d_{k-1}, d_k] of each node's stage with
 * lattice-masked attention, the shared exit head (final RMSNorm + LM head) over all
 * nodes, DECS, and the host-side commit that decides the next round.
 *
 * Conventions
 *  - Every entry point returns DEX_OK (0) or a negative dex_status; dex_strerror()
 *    names it.  A failing call leaves the handle usable unless it returns DEX_ECUDA.
 *  - "device" pointers are CUDA global-memory addresses on the handle's device;
 *    "host" pointers are ordinary process memory.  Weights are bf16, row-major
 *    [out_features][in_features], and stay owned by the caller, who keeps them alive
 *    until dex_free().  The library owns its KV caches and workspaces, allocated in
 *    dex_init() and released by dex_free().
 *  - Arithmetic: bf16 weights on the tensor cores with fp32 accumulation; activations
 *    enter every GEMM as a pair of bf16 operands (x ~= hi + lo, about 17 significant
 *    bits), hidden states are fp32, and the K/V caches hold fp16 (11 significant bits,
 *    8x finer than bf16 at the same two bytes) read into fp32 attention arithmetic.
 *  - All work is issued on the stream given to dex_init().  Calls returning host data
 *    synchronise that stream.  A handle is not thread-safe.
 *  - Positions are absolute token indices starting at 0; the commit position p_c is
 *    the index of the next token to be committed.
 */
#ifndef DEX_H_
#define DEX_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dex_status {
  DEX_OK = 0,
  DEX_EINVAL = -1,     /* a bad argument (null pointer, size out of range, unsupported shape) */
  DEX_ENOMEM = -2,     /* device or host allocation failed */
  DEX_ECUDA = -3,      /* a CUDA runtime or driver call failed; the handle should be freed */
  DEX_ECAPACITY = -4,  /* a sequence would exceed max_ctx or max_new */
  DEX_ETIMEOUT = -5,   /* a bounded device wait gave up (kernel reported a stalled pipeline) */
  DEX_ESTATE = -6,     /* call out of order (e.g. dex_step before dex_prefill) */
  DEX_ENODEV = -7,     /* no usable sm_103 device */
  DEX_ERANGE = -8      /* a linear layer's split-K partial sum was not finite or reached 2^30 in
                          magnitude (the range of the exact fixed-point segment sum); the
                          round's results are void, the handle stays usable */
} dex_status;

/* Model description (Llama-style pre-norm decoder, no biases, SwiGLU FFN, RoPE).
 * The residual-branch scale of the method's synthetic models is expected folded
 * into wo and wd.  layers points to a HOST array of n_layers * 9 DEVICE pointers,
 * per layer in the order: attn_norm[d], wq[H*hd][d], wk[KVH*hd][d], wv[KVH*hd][d],
 * wo[d][H*hd], ffn_norm[d], wg[d_ff][d], wu[d_ff][d], wd[d][d_ff].  The array is
 * copied by dex_init().  Constraints: d_model % 128 == 0 and <= 8192, head_dim in {64, 128},
 * n_heads % n_kv_heads == 0, n_heads*head_dim and n_kv_heads*head_dim multiples of 128,
 * d_ff a multiple of 8 (>= 64), every weight 16-byte aligned (DEX_EINVAL otherwise). */
typedef struct dex_model {
  int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, d_ff, vocab;
  float rms_eps, rope_theta;
  const void* embed;        /* device, [vocab][d_model] bf16 */
  const void* final_norm;   /* device, [d_model] bf16 */
  const void* lm_head;      /* device, [vocab][d_model] bf16 (== embed for a tied head) */
  const void* const* layers;/* host array of n_layers*9 device pointers (see above) */
  /* Inducing adapters (Appendix C.2), or NULL: a host array of (n_X - 1) * 5 device pointers,
   * one adapter per non-final depth X[k], k < n_X - 1, of the X given to dex_init, in the
   * order g[d] (RMSNorm gain), w1[2d][d], b1[2d], w2[d][2d], b2[d] (bf16), with
   * adapter_alpha a host array of the n_X - 1 scalar gates.  The node of a non-final stage
   * is decoded from h + alpha (w2 SiLU(w1 RMSNorm(h; g) + b1) + b2); the final depth never is. */
  const void* const* adapters;
  const float* adapter_alpha;
} dex_model;

/* Decode setup.  sample=0: greedy (ties -> lowest id); sample=1: Gumbel-max at
 * temperature tau with noise rows keyed by (seed, sequence, target position).
 * decs=1 enables DECS masking (Algorithm 2); decs=0 decodes every node
 * independently.  debug_logits=1 keeps the fp32 logits of the last round's nodes
 * for dex_debug_logits() (costs vocab*4 bytes per node of device memory). */
typedef struct dex_decode_cfg {
  int32_t batch;        /* independent sequences, 1..64 */
  int32_t max_ctx;      /* capacity in positions per sequence (prompt + new + N), <= 4096 */
  int32_t max_new;      /* tokens to commit per sequence */
  int32_t sample;
  float tau;
  uint64_t seed;
  int32_t decs;
  int32_t debug_logits;
  int32_t max_branch;   /* 0: the full lattice; k > 0: a sparse lattice whose nodes speculate at
                           most k tokens ahead of the commit (k position moves on their path;
                           the final-depth commit, hence the token stream, is unchanged) */
} dex_decode_cfg;

typedef struct dex_handle dex_handle;

/* Create a handle for exploration set X = {d_0 < ... < d_{N-1} = n_layers}
 * (Definition 4), 1 <= N <= 10.  stream: a cudaStream_t (NULL = legacy default).
 * Allocates every device buffer the decode needs.  Errors: DEX_EINVAL for a bad
 * model/X/cfg, DEX_ENODEV, DEX_ENOMEM, DEX_ECUDA. */
int dex_init(const dex_model* model, const int32_t* X, int32_t n_X, const dex_decode_cfg* cfg,
             void* stream, dex_handle** out);

/* init(x, {E_k}) of Algorithm 1 for sequence seq: writes the committed KV cache of
 * prompt positions 0..n_tokens-2 and makes the last prompt token the root input
 * (state q = 0, empty explore buffer).  tokens: HOST int32 [n_tokens], n_tokens >= 1,
 * ids in [0, vocab).  Resets the sequence's decode state. */
int dex_prefill(dex_handle* h, int32_t seq, const int32_t* tokens, int32_t n_tokens);

/* One DEX round over every prefilled, unfinished sequence: expand the level-q nodes,
 * exit head + DECS, insert, and -- for sequences whose anchor reached the final
 * depth -- validate_and_commit and collapse.  out_tokens / n_committed: HOST int32
 * [batch]; n_committed[b] is 1 when sequence b committed out_tokens[b] this round,
 * else 0.  Returns DEX_ESTATE when no sequence is active. */
int dex_step(dex_handle* h, int32_t* out_tokens, int32_t* n_committed);

/* Run dex_step until every prefilled sequence has committed max_new tokens.
 * out: HOST int32 [batch][max_new]; rows of sequences never prefilled are left as is. */
int dex_generate(dex_handle* h, int32_t* out);

/* Plain autoregressive round on the same kernels (one node per sequence through all
 * layers, exit at the final depth): the lossless reference DEX must equal.  Same
 * outputs as dex_step.  Must not be mixed with dex_step on a sequence between two
 * dex_prefill calls (DEX_ESTATE). */
int dex_ar_step(dex_handle* h, int32_t* out_tokens, int32_t* n_committed);

/* Run dex_ar_step until every prefilled sequence has max_new tokens; out as dex_generate. */
int dex_ar_generate(dex_handle* h, int32_t* out);

/* Counters since dex_init / the last dex_reset_stats. */
typedef struct dex_stats {
  int64_t rounds;           /* rounds executed (DEX or AR) */
  int64_t commits;          /* committed tokens over all sequences */
  int64_t nodes;            /* lattice nodes evaluated */
  int64_t max_round_nodes;  /* largest single-round node batch */
  int64_t layer_passes;     /* sum over rounds of d of the deepest live stage */
  int64_t node_layers;      /* sum over nodes of the layer count of their stage */
  int64_t depth_charge;     /* sum over committed tokens of d_{k*} (Eq. 12's W) */
  int64_t kstar_hist[16];   /* committed tokens by accepted branch k* */
  int64_t weight_bytes;     /* algorithmic weight bytes streamed (each live layer once per round) */
  int64_t kv_bytes;         /* algorithmic committed + branch KV bytes read */
  int64_t h2d_bytes, d2h_bytes;
  int64_t kernel_launches;
  int64_t gemm_launches;    /* linear-layer GEMM launches (the dominant kernel) */
  int64_t gemm_bytes;       /* their algorithmic bytes (weights + activations in/out) */
  double ms_gemm;           /* summed CUDA-event duration of those launches (timing >= 2) */
  double ms_expand, ms_exit, ms_collapse, ms_host;  /* phase split (timing >= 1) */
  int64_t attn_launches;    /* lattice-attention launches */
  double ms_attn;           /* summed CUDA-event duration of those launches (timing >= 2) */
} dex_stats;

int dex_get_stats(const dex_handle* h, dex_stats* out);
int dex_reset_stats(dex_handle* h);

/* timing: 0 off; 1 = CUDA events around the expansion / exit+DECS / collapse phases of
 * each round; 2 = also around every linear-layer GEMM and attention launch (adds events,
 * which also stop programmatic-dependent-launch overlap across them); 3 = level 1
 * plus per-CTA clock records of the GEMM launches that follow (diagnostics: only when the
 * environment variable DEX_TIMELINE names a file, which dex_free() writes; the first
 * DEX_TIMELINE_LAUNCHES launches, default 512, are kept). */
int dex_set_timing(dex_handle* h, int32_t level);

/* Lattice nodes of the most recent round, in evaluation order: HOST int32
 * [max_rows][8] = {seq, heap index, stage, plen, target position, token, prior
 * count, input position}.  *rows_out receives the number of nodes. */
int dex_last_round_nodes(const dex_handle* h, int32_t* host_out, int32_t max_rows, int32_t* rows_out);

/* fp32 logits of the most recent round's nodes (same order as dex_last_round_nodes),
 * before masking and noise.  Needs cfg.debug_logits = 1.  host_out: HOST float
 * [max_rows][vocab]. */
int dex_debug_logits(dex_handle* h, float* host_out, int32_t max_rows, int32_t* rows_out);

const char* dex_strerror(int code);
void dex_free(dex_handle* h);

/* Failure-path self-test (diagnostics; the paper has no counterpart).  Runs the bounded
 * mbarrier wait that every pipeline of the library uses against a barrier that nothing
 * completes, with a limit of limit_us microseconds (1..1000000), on the handle's stream,
 * and reads the device error flag back exactly as a decode round does.  Returns
 * DEX_ETIMEOUT when the wait gave up as designed (the flag is then cleared and the handle
 * stays usable), DEX_OK if it did not, DEX_EINVAL for a bad argument.  Synchronises the
 * stream.  Allocation failures of dex_init can likewise be injected on the host: with the
 * environment variable DEX_FAIL_ALLOC_AT=k set, the k-th device or pinned-host allocation
 * of dex_init reports failure, and dex_init returns DEX_ENOMEM after releasing everything
 * it had allocated. */
int dex_selftest_stall(dex_handle* h, int32_t limit_us);

/* ---- kernels in isolation ------------------------------------------------------ */

/* One node of an isolated exit-head + DECS call. */
typedef struct dex_exit_node {
  int32_t seq;          /* sequence id (Gumbel row key) */
  int32_t target_pos;   /* absolute position being predicted (Gumbel row key) */
  int32_t unmasked;     /* 1 for the final-depth reference: no DECS mask */
  int32_t prior_off;    /* first prior token in the priors array */
  int32_t n_prior;      /* number of prior tokens (shallower proposals of the slot chain) */
} dex_exit_node;

/* Exit head + DECS over n nodes (section 3.3, Appendix C.1 Algorithm 2, exit head of
 * Appendix C.2): token[i] = argmax_v score_i(v), with logits z = RMSNorm(h_i; g) W^T,
 * score = -inf for masked priors, else z (greedy) or z / tau + G(seed, seq, pos, v).
 * h: device bf16 [n][d]; final_norm: device bf16 [d]; lm_head: device bf16
 * [vocab][d]; nodes: device [n]; priors: device int32; tokens: device int32 [n];
 * logits: device fp32 [n][vocab] or NULL.  1 <= n <= 256, d % 128 == 0, d <= 8192.
 * Allocates its scratch with the stream-ordered allocator; stream-ordered, no sync, so
 * device-side failures cannot be returned: if a bounded wait inside the GEMM gives up
 * (the decoder would report DEX_ETIMEOUT), every token of the call is written as -1. */
int dex_exit_head_decs(const void* h, int32_t n, int32_t d, const void* final_norm, float rms_eps,
                       const void* lm_head, int32_t vocab, const dex_exit_node* nodes,
                       const int32_t* priors, int32_t sample, float tau, uint64_t seed,
                       int32_t* tokens, float* logits, void* stream);

/* Size of the fixed device scratch of dex_exit_head_decs_noalloc: 32 MiB per GPU. */
#define DEX_NOALLOC_SCRATCH_BYTES (32u << 20)

/* The exit head + DECS of dex_exit_head_decs, for callers that must not allocate device
 * memory during the call (for example code running under another component's stream
 * capture or allocator, or with a memory budget fixed at start-up).  The paper has no
 * counterpart: this is a deployment convenience of this library.
 * It runs the GEMM on one CTA per SM (a deeper weight ring; its split-K partials then fit
 * the fixed scratch) where dex_exit_head_decs uses two, so the k-segment split and hence
 * the last bits of the logits may differ between the two entry points; each is within the
 * same tolerance of the fp64 exit head, and tokens agree wherever the decision margin is
 * not within rounding of zero.  A stalled bounded wait writes every token as -1, as in
 * dex_exit_head_decs (the stall flag lives in the scratch and is cleared by the next call).
 * Scratch comes from one file-scope device array of DEX_NOALLOC_SCRATCH_BYTES that every
 * GPU loading the library keeps until the process exits; no cudaMalloc/cudaFree or other
 * allocating routine is called.  The array's device address is looked up on the first call
 * made on each device (with that device current), so make that first call before any
 * stream capture.  Calls share the array: calls that may overlap on the GPU (different
 * streams, or several host threads) race and must be serialised by the caller.  Returns
 * DEX_ECAPACITY, doing nothing, when the call's scratch (hidden tile, RMSNorm partials,
 * split-K partials) would exceed DEX_NOALLOC_SCRATCH_BYTES; other arguments and errors as
 * dex_exit_head_decs. */
int dex_exit_head_decs_noalloc(const void* h, int32_t n, int32_t d, const void* final_norm, float rms_eps,
                               const void* lm_head, int32_t vocab, const dex_exit_node* nodes,
                               const int32_t* priors, int32_t sample, float tau, uint64_t seed,
                               int32_t* tokens, float* logits, void* stream);

/* Geometry of the KV caches used by dex_kv_collapse.  committed: [batch][n_layers][2]
 * [n_kv_heads][max_ctx][head_dim] bf16; pool: [batch][n_slots][n_layers][2]
 * [n_kv_heads][head_dim] bf16 (one slot per sampling-slot chain). */
typedef struct dex_kv_geom {
  int32_t batch, n_layers, n_kv_heads, head_dim, max_ctx, n_slots;
} dex_kv_geom;

/* Copy the branch KV of a surviving slot chain into the committed cache at its
 * position (the collapse of section 3.2 for the new anchor path). */
typedef struct dex_copy_job {
  int32_t seq, slot, pos, n_layers;   /* layers 0..n_layers-1 of slot -> position pos */
} dex_copy_job;

/* Vectorised gather/scatter of n_jobs copy jobs (device array, 0 <= n_jobs <= 65535).
 * committed / pool: device, 16-byte aligned, with geom's layouts; head_dim a multiple of 8.
 * A job with seq outside [0, batch), slot outside [0, n_slots), pos outside [0, max_ctx) or
 * n_layers outside [1, n_layers] is skipped without any memory access.  rejected: device
 * int32 or NULL; when given, the call zeroes it (stream-ordered) and adds one per skipped
 * job.  Stream-ordered, no sync.  DEX_EINVAL for a bad geometry or pointer. */
int dex_kv_collapse(void* committed, const void* pool, const dex_kv_geom* geom,
                    const dex_copy_job* jobs, int32_t n_jobs, int32_t* rejected, void* stream);

/* ---- host-only lattice scheduler (no GPU needed) ---------------------------------- */

/* One planned lattice node (HOST struct). */
typedef struct dex_plan_node {
  int32_t seq, heap, stage, plen;
  int32_t pos;          /* position of the node's input token: p_c - 1 + plen */
  int32_t c_end;        /* keys at positions < c_end come from the committed cache */
  int32_t slot;         /* pool slot of the node's slot chain */
  int32_t kv_commit;    /* 1 for the anchor path: K/V written to the committed cache */
  int32_t token;        /* input token for stage-0 nodes, -1 for depth children */
  int32_t target_pos;   /* p_c + plen */
  int32_t unmasked;     /* 1 for the final-depth reference node */
  int32_t n_prior, n_tail;
  int32_t prior[16];    /* DECS priors: tokens of shallower nodes in the slot chain */
  int32_t tail[16];     /* pool slots holding the KV of positions c_end .. pos */
} dex_plan_node;

typedef struct dex_lattice dex_lattice;

int dex_lattice_new(const int32_t* X, int32_t n_X, int32_t batch, int32_t decs, int32_t max_branch,
                    dex_lattice** out);
/* Start sequence seq with p_c committed tokens, last_token at position p_c - 1. */
int dex_lattice_start(dex_lattice* lat, int32_t seq, int32_t p_c, int32_t last_token);
/* Nodes of the next round (level q of each active sequence), grouped by stage. */
int dex_lattice_plan(dex_lattice* lat, dex_plan_node* out, int32_t max_nodes, int32_t* n_nodes);
/* Insert the planned nodes' tokens; commit and collapse where the anchor reached the
 * final depth.  committed: HOST int32 [batch] (-1 = none); kstar: HOST int32 [batch]
 * (-1 = none); jobs: copy jobs the collapse needs (n_jobs <= max_jobs). */
int dex_lattice_update(dex_lattice* lat, const int32_t* tokens, int32_t* committed, int32_t* kstar,
                       dex_copy_job* jobs, int32_t max_jobs, int32_t* n_jobs);
/* State of sequence seq: {q, p_c, slots in use}. */
int dex_lattice_state(const dex_lattice* lat, int32_t seq, int32_t* q, int32_t* p_c, int32_t* slots_used);
void dex_lattice_free(dex_lattice* lat);

#ifdef __cplusplus
}
#endif
#endif /* DEX_H_ */

// Small kernels of a DEX round: stage-input assembly (embedding gather for stage-0
// nodes, hidden-state hand-over for depth children), the KV collapse gather/scatter
// that moves the new anchor path's branch KV into the committed cache, and the input
// preparation / token decode of an isolated exit-head call.
#include "common.cuh"
#include "kernels.h"

#include <stdlib.h>

namespace dex {

// Sums of squares of the d/128 feature tiles of one row, one value per thread per tile
// (thread t holds feature 128 i + t of tile i), in the canonical order shared with the
// residual epilogue of the GEMM: per-warp butterfly (warp_sum), then (q0 + q1) + (q2 + q3)
// over the four warps.  A row's RMSNorm scale therefore does not depend on which kernel
// produced its partial sums.  ssq_out: [ndt] (written by threads 0..ndt-1).
template <int MAXT>
__device__ __forceinline__ void row_tile_ssq(const float (&x)[MAXT], int ndt, float* qbuf, float* ssq_out) {
  const int warp = threadIdx.x >> 5;
#pragma unroll
  for (int t = 0; t < MAXT; ++t) {
    if (t < ndt) {
      const float s = warp_sum(__fmul_rn(x[t], x[t]));
      if ((threadIdx.x & 31) == 0) qbuf[t * 4 + warp] = s;
    }
  }
  __syncthreads();
  if (static_cast<int>(threadIdx.x) < ndt) {
    const float* q = qbuf + threadIdx.x * 4;
    ssq_out[threadIdx.x] = __fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3]));
  }
}

constexpr int kMaxTiles = 64;   // d_model up to 8192

// One CTA (128 threads) per node row.  Stage-0 nodes start a slot chain: h = E[token]
// into the chain's hidden row.  Depth children continue the chain's hidden row left by
// the previous stage.  Writes the first layer's input h * g as a hi/lo bf16 pair and the
// RMSNorm partial sums, and clears the row's exit-head argmax slot.  The whole row is loaded
// before any reduction so the loads overlap.
__global__ void __launch_bounds__(128) assemble_kernel(const AssembleArgs a) {
  __shared__ float qbuf[kMaxTiles * 4];
  const int row = blockIdx.x;
  griddep_wait();
  griddep_launch_dependents();
  const DevNode nd = a.nodes[row];
  if (a.best && threadIdx.x == 0) a.best[row] = 0ull;
  const __nv_bfloat16* g = a.attn_norm[nd.first_layer];
  float* hrow = a.hidden + static_cast<size_t>(nd.hrow) * a.d;
  const int ndt = a.d / 128;
  float x[kMaxTiles];
#pragma unroll
  for (int t = 0; t < kMaxTiles; ++t) {
    if (t < ndt) {
      const int f = t * 128 + threadIdx.x;
      x[t] = nd.token >= 0 ? bf16_to_f32(a.embed[static_cast<size_t>(nd.token) * a.d + f]) : hrow[f];
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxTiles; ++t) {
    if (t < ndt) {
      const int f = t * 128 + threadIdx.x;
      if (nd.token >= 0) hrow[f] = x[t];
      const size_t o = static_cast<size_t>(row) * a.d + f;
      store_pair(a.hb + o, a.hb + static_cast<size_t>(a.plane_rows) * a.d + o, __fmul_rn(x[t], bf16_to_f32(g[f])));
    }
  }
  row_tile_ssq<kMaxTiles>(x, ndt, qbuf, a.ssq + static_cast<size_t>(row) * ndt);
}

int smem_carveout_pref() {
  static const int pref = [] {
    const char* e = getenv("DEX_SMEM_CARVEOUT");
    if (!e) return -1;
    const int v = atoi(e);
    return (v >= 0 && v <= 100) ? v : -1;
  }();
  return pref;
}

cudaError_t launch_assemble(const AssembleArgs& a, cudaStream_t st, bool pdl) {
  if (a.n_rows <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = apply_carveout(assemble_kernel);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (!a.nodes || !a.embed || !a.attn_norm || !a.hidden || !a.hb || !a.ssq || a.d % 128 || a.d > 128 * 64 ||
      a.plane_rows < a.n_rows)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.n_rows));
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, assemble_kernel, a);
}

// Collapse gather/scatter: for each job, layers 0..n_layers-1 of the slot chain's branch
// KV (contiguous [layer][2][KVH] head rows in the pool) go to position pos of the
// committed cache.  16-byte vectors; consecutive threads cover consecutive bytes of a
// head row on both sides.
__global__ void __launch_bounds__(256) collapse_kernel(const CollapseArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const CopyJob job = a.jobs[blockIdx.y];
  if (job.seq < 0 || job.seq >= a.batch || job.slot < 0 || job.slot >= a.n_slots || job.pos < 0 ||
      job.pos >= a.max_ctx || job.n_layers < 1 || job.n_layers > a.L) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      if (a.err) atomicExch(a.err, DEV_BAD_INDEX);
      if (a.rejected) atomicAdd(a.rejected, 1);
    }
    return;
  }
  const int vec_per_row = a.row_bytes / 16;
  const int total = job.n_layers * 2 * a.KVH * vec_per_row;
  const uint4* src = reinterpret_cast<const uint4*>(a.kv_pool) +
                     (static_cast<size_t>(job.seq) * a.n_slots + job.slot) * a.L * 2 * a.KVH * vec_per_row;
  uint4* commit = reinterpret_cast<uint4*>(a.kv_commit);
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
    const int ch = idx % vec_per_row;
    int rest = idx / vec_per_row;
    const int h = rest % a.KVH;
    rest /= a.KVH;
    const int kv = rest & 1, layer = rest >> 1;
    commit[((((static_cast<size_t>(job.seq) * a.L + layer) * 2 + kv) * a.KVH + h) * a.max_ctx + job.pos) *
               vec_per_row + ch] = src[idx];
  }
}

cudaError_t launch_collapse(const CollapseArgs& a, cudaStream_t st, bool pdl) {
  if (a.n_jobs <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = apply_carveout(collapse_kernel);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (!a.jobs || !a.kv_commit || !a.kv_pool || a.row_bytes < 16 || a.row_bytes % 16 || a.batch < 1 || a.L < 1 ||
      a.KVH < 1 || a.max_ctx < 1 || a.n_slots < 1 ||
      (reinterpret_cast<uintptr_t>(a.kv_commit) & 15) || (reinterpret_cast<uintptr_t>(a.kv_pool) & 15))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(32, static_cast<unsigned>(a.n_jobs));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, collapse_kernel, a);
}

// Isolated exit head: bf16 hidden rows -> the hi/lo pair of h * g and the RMSNorm
// partial sums.
__global__ void __launch_bounds__(128) exit_prep_kernel(const __nv_bfloat16* h, int d, const __nv_bfloat16* g,
                                                        __nv_bfloat16* hb, int plane_rows, float* ssq,
                                                        unsigned long long* best) {
  __shared__ float qbuf[kMaxTiles * 4];
  const int row = blockIdx.x;
  if (threadIdx.x == 0) best[row] = 0ull;
  const int ndt = d / 128;
  float x[kMaxTiles];
#pragma unroll
  for (int t = 0; t < kMaxTiles; ++t)
    if (t < ndt) x[t] = bf16_to_f32(h[static_cast<size_t>(row) * d + t * 128 + threadIdx.x]);
#pragma unroll
  for (int t = 0; t < kMaxTiles; ++t) {
    if (t < ndt) {
      const int f = t * 128 + threadIdx.x;
      const size_t o = static_cast<size_t>(row) * d + f;
      store_pair(hb + o, hb + static_cast<size_t>(plane_rows) * d + o, __fmul_rn(x[t], bf16_to_f32(g[f])));
    }
  }
  row_tile_ssq<kMaxTiles>(x, ndt, qbuf, ssq + static_cast<size_t>(row) * ndt);
}

cudaError_t launch_exit_prep(const __nv_bfloat16* h, int n, int d, const __nv_bfloat16* g, __nv_bfloat16* hb,
                             int plane_rows, float* ssq, unsigned long long* best, cudaStream_t st) {
  if (n < 1 || plane_rows < n || d % 128 || d > 128 * kMaxTiles || !h || !g || !hb || !ssq || !best)
    return cudaErrorInvalidValue;
  exit_prep_kernel<<<n, 128, 0, st>>>(h, d, g, hb, plane_rows, ssq, best);
  return cudaGetLastError();
}

// Weight packing (once per handle): one thread per 16-byte chunk of the packed image.
__global__ void __launch_bounds__(256) pack_kernel(int mode, PackSrc s0, PackSrc s1, PackSrc s2, int K, int kblocks,
                                                   long long n_chunks, uint8_t* out) {
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n_chunks;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx & 7), r = static_cast<int>((idx >> 3) & 127);
    const long long box = idx >> 10;
    const int t = static_cast<int>(box / kblocks), k = static_cast<int>(box % kblocks);
    const __nv_bfloat16* src = nullptr;
    int srow = 0;
    if (mode == PACK_SWIGLU) {
      const PackSrc& ps = r < 64 ? s0 : s1;
      srow = t * 64 + (r & 63);
      if (srow < ps.rows) src = ps.ptr;
    } else {
      int grow = t * 128 + r;
      if (grow < s0.rows) {
        src = s0.ptr;
        srow = grow;
      } else if ((grow -= s0.rows) < s1.rows) {
        src = s1.ptr;
        srow = grow;
      } else if ((grow -= s1.rows) < s2.rows) {
        src = s2.ptr;
        srow = grow;
      }
    }
    const int col = k * 64 + ((c ^ (r & 7)) * 8);   // the chunk stored at position c
    uint4 v = make_uint4(0, 0, 0, 0);
    if (src && col < K) v = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(srow) * K + col);
    *reinterpret_cast<uint4*>(out + box * 16384 + r * 128 + c * 16) = v;
  }
}

size_t packed_bytes(int n_tiles, int kblocks) { return static_cast<size_t>(n_tiles) * kblocks * 16384; }

cudaError_t launch_pack(int mode, PackSrc s0, PackSrc s1, PackSrc s2, int K, int n_tiles, uint8_t* out,
                        cudaStream_t st) {
  if (K % 8) return cudaErrorInvalidValue;
  const int kblocks = (K + 63) / 64;
  const long long n_chunks = static_cast<long long>(n_tiles) * kblocks * 1024;
  const long long blocks = (n_chunks + 255) / 256;
  pack_kernel<<<static_cast<unsigned>(blocks < 65535 * 16 ? blocks : 65535 * 16), 256, 0, st>>>(
      mode, s0, s1, s2, K, kblocks, n_chunks, out);
  return cudaGetLastError();
}

__global__ void decode_best_kernel(const unsigned long long* best, int n, const int32_t* err, int32_t* tokens) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  tokens[i] = (err && *err) ? -1 : static_cast<int32_t>(~static_cast<uint32_t>(best[i] & 0xffffffffull));
}

static cudaError_t launch_plain(const void* func, int grid, int block, void** args, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.stream = st;
  return cudaLaunchKernelExC(&cfg, func, args);
}

cudaError_t launch_decode_best(const unsigned long long* best, int n, const int32_t* err, int32_t* tokens,
                               cudaStream_t st) {
  if (n < 1 || !best || !tokens) return cudaErrorInvalidValue;
  void* args[] = {&best, &n, &err, &tokens};
  return launch_plain(reinterpret_cast<const void*>(decode_best_kernel), (n + 127) / 128, 128, args, st);
}

// The public node struct of an isolated exit-head call: five int32 fields
// (seq, target_pos, unmasked, prior_off, n_prior).
__global__ void exit_nodes_kernel(const int32_t* in, int n, DevNode* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  DevNode d = {};
  d.seq = in[5 * i + 0];
  d.target_pos = in[5 * i + 1];
  d.unmasked = in[5 * i + 2];
  d.prior_off = in[5 * i + 3];
  d.n_prior = in[5 * i + 4];
  out[i] = d;
}

cudaError_t launch_exit_nodes(const void* exit_nodes, int n, DevNode* out, cudaStream_t st) {
  if (n < 1 || !exit_nodes || !out) return cudaErrorInvalidValue;
  const int32_t* in = static_cast<const int32_t*>(exit_nodes);
  void* args[] = {&in, &n, &out};
  return launch_plain(reinterpret_cast<const void*>(exit_nodes_kernel), (n + 127) / 128, 128, args, st);
}

}  // namespace dex

// cache_append.cu -- the rows of a batch's new tokens into a row cache.
//
// Before the lightning indexer scores a new token, the token's own indexer
// key and its latent row (one per layer) must sit in the caches: its causal
// context includes itself, and the top-k selector reads the whole context from
// HBM ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", What it claims /
// Model).  Query token t of sequence b (position p_t) writes its row into the
// pool row that holds token p_t of b: page_table[b, p_t / 64] * 64 + p_t % 64
// for a paged cache, seq_start[b] + p_t for a contiguous one.
//
// One warp per token, 16-byte copies; the per-call plan (sequence and position
// of every query) comes from the plan kernel launched just before.
#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kWarps = 8;

struct AppendParams {
  const __nv_bfloat16* src;
  int64_t ld_src;
  CacheView c;
  int32_t row_elems;
  int32_t T;
  const int32_t* q_seq;
  const int32_t* q_n;
  int* err;
};

__global__ void __launch_bounds__(32 * kWarps) cache_append_kernel(AppendParams p) {
  pdl_wait();  // the plan (previous grid) is complete from here on
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + warp;
  if (t >= p.T) return;
  const int n = p.q_n[t];  // p_t + 1, or 0 when the token's sequence is malformed (flagged by the plan)
  if (n <= 0) return;
  const int64_t row = cache_row(p.c, p.q_seq[t], n - 1);
  if (row < 0) {
    if (lane == 0) atomicOr(p.err, DEV_ERR_BAD_INDEX);
    return;
  }
  const uint4* s = reinterpret_cast<const uint4*>(p.src + (int64_t)t * p.ld_src);
  uint4* d = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(p.c.base) + row * p.c.row_stride);
  for (int i = lane; i < p.row_elems / 8; i += 32) d[i] = __ldg(s + i);
}

}  // namespace

cudaError_t launch_cache_append(const AppendLaunch& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  AppendParams p;
  p.src = static_cast<const __nv_bfloat16*>(a.src);
  p.ld_src = a.ld_src;
  p.c = a.c;
  p.row_elems = a.row_elems;
  p.T = a.T;
  p.q_seq = a.q_seq;
  p.q_n = a.q_n;
  p.err = a.err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.T + kWarps - 1) / kWarps, 1, 1);
  cfg.blockDim = dim3(32 * kWarps, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute at = pdl_attribute();
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cache_append_kernel, p);
}

}  // namespace dsa

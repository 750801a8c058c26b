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
// One warp per token, 16-byte copies.  A warp finds its token's sequence by a
// binary search of cu_seqlens_q and checks that sequence's lengths itself, so
// the call is one launch with no per-call plan ahead of it (a decode step
// appends the indexer key and every layer's latent row: one small launch
// each).
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
  int32_t B;
  int32_t max_seqlen_k;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens_k;
  int* err;
};

__global__ void __launch_bounds__(32 * kWarps) cache_append_kernel(AppendParams p) {
  pdl_wait();  // rows or lengths written by the previous grid are visible from here on
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + warp;
  if (t >= p.T) return;
  int lo = 0, hi = p.B - 1;  // last b with cu_seqlens_q[b] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_seqlens_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int c0 = __ldg(p.cu_seqlens_q + lo), c1 = __ldg(p.cu_seqlens_q + lo + 1);
  const int len = __ldg(p.seq_lens_k + lo);
  const int nq = c1 - c0, i = t - c0;
  // the same checks as the forward's plan: a malformed sequence writes nothing
  if (c0 < 0 || nq < 0 || c1 > p.T || len < nq || len > p.max_seqlen_k || i < 0 || i >= nq) {
    if (lane == 0) atomicOr(p.err, DEV_ERR_BAD_INDEX);
    return;
  }
  const int64_t row = cache_row(p.c, lo, len - nq + i);  // token position p_t = len - nq + i
  if (row < 0) {
    if (lane == 0) atomicOr(p.err, DEV_ERR_BAD_INDEX);
    return;
  }
  const uint4* s = reinterpret_cast<const uint4*>(p.src + (int64_t)t * p.ld_src);
  uint4* d = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(p.c.base) + row * p.c.row_stride);
  for (int k = lane; k < p.row_elems / 8; k += 32) d[k] = __ldg(s + k);
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
  p.B = a.B;
  p.max_seqlen_k = a.max_seqlen_k;
  p.cu_seqlens_q = a.cu_seqlens_q;
  p.seq_lens_k = a.seq_lens_k;
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

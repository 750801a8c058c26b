// plan.cu -- per-call plan of a ragged batch: sequence and causal length of
// every query token, and the indexer's flat list of (query group, 128-key
// tile) work items.  One block; runs ahead of the compute kernels on the same
// stream, so no host round trip is needed to size ragged work.
#include "internal.cuh"

namespace dsa {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kMaxSeqs = 16384;  // sequence offsets kept in shared memory

// Exclusive block-wide scan of one int per thread; returns the prefix and
// writes the block total to *total.  All threads of the block must call it.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

__device__ __forceinline__ bool seq_ok(const PlanParams& p, int b, int* nq_out, int* len_out) {
  const int c0 = __ldg(p.cu_seqlens_q + b), c1 = __ldg(p.cu_seqlens_q + b + 1);
  const int len = __ldg(p.seq_lens_k + b);
  const int nq = c1 - c0;
  *nq_out = nq;
  *len_out = len;
  return c0 >= 0 && nq >= 0 && c1 <= p.T && len >= nq && len <= p.max_seqlen_k;
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanParams p) {
  extern __shared__ int goff[];  // [B + 1] group offsets of the sequences
  __shared__ int warp_sums[32];
  __shared__ int s_total;
  const int G = p.group;

  // (1) groups per sequence, and their offsets
  int running = 0;
  for (int b0 = 0; b0 < p.B; b0 += kPlanThreads) {
    const int b = b0 + threadIdx.x;
    int ng = 0;
    if (b < p.B) {
      int nq, len;
      if (seq_ok(p, b, &nq, &len)) {
        ng = (nq + G - 1) / G;
      } else {
        atomicOr(p.err, DEV_ERR_BAD_INDEX);
      }
    }
    int tot;
    const int ex = block_exclusive_scan(ng, warp_sums, &tot);
    if (b < p.B) goff[b] = running + ex;
    running += tot;
  }
  if (threadIdx.x == 0) goff[p.B] = running;
  const int n_groups = running;
  __syncthreads();

  // (2) every query: its sequence and causal context length
  for (int t = threadIdx.x; t < p.T; t += kPlanThreads) {
    int lo = 0, hi = p.B - 1;  // last b with cu[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.cu_seqlens_q + mid) <= t) lo = mid; else hi = mid - 1;
    }
    int nq, len;
    const bool ok = seq_ok(p, lo, &nq, &len);
    const int i = t - __ldg(p.cu_seqlens_q + lo);
    p.plan.q_seq[t] = lo;
    p.plan.q_n[t] = (ok && i >= 0 && i < nq) ? (len - nq + i + 1) : 0;
  }

  // (3) every group: its queries and its number of 128-key work items
  running = 0;
  for (int g0 = 0; g0 < n_groups; g0 += kPlanThreads) {
    const int g = g0 + threadIdx.x;
    int items = 0;
    if (g < n_groups) {
      int lo = 0, hi = p.B - 1;  // last b with goff[b] <= g
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (goff[mid] <= g) lo = mid; else hi = mid - 1;
      }
      const int b = lo;
      const int j = g - goff[b];
      int nq, len;
      seq_ok(p, b, &nq, &len);
      const int q0 = __ldg(p.cu_seqlens_q + b) + j * G;
      const int cnt = min(G, nq - j * G);
      const int n_last = len - nq + j * G + cnt;  // causal n of the group's last query
      p.plan.g_info[g] = make_int4(b, q0, cnt, n_last);
      items = (n_last > p.skip_dense_k) ? (n_last + kIdxTileKeys - 1) / kIdxTileKeys : 0;
    }
    int tot;
    const int ex = block_exclusive_scan(items, warp_sums, &tot);
    if (g < n_groups) p.plan.g_tile_start[g] = running + ex;
    running += tot;
  }
  if (threadIdx.x == 0) {
    p.plan.g_tile_start[n_groups] = running;
    p.plan.header[0] = n_groups;
    p.plan.header[1] = running;
  }
}

}  // namespace

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
  if (p.B > kMaxSeqs) return cudaErrorInvalidValue;
  const size_t smem = sizeof(int) * (size_t)(p.B + 1);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  plan_kernel<<<1, kPlanThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa

// plan.cu -- per-call plan of a ragged batch: sequence and causal length of
// every query token (in cache entries: tokens, or complete blocks of `ratio`
// tokens), and the indexer's flat list of (query group, 128-key tile) work
// items.  One block; runs ahead of the compute kernels on the same
// stream, so no host round trip is needed to size ragged work.  The batch's
// two length arrays are staged in shared memory so every search is on-chip.
#include "internal.cuh"

namespace dsa {

namespace {

constexpr int kPlanThreads = 1024;  // the most threads; a small batch is planned by fewer
constexpr int kMaxSeqs = 16384;  // cu_seqlens, lengths and group offsets kept in shared memory

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
    int s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
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

struct SeqArrays {
  const int* cu;   // [B + 1]
  const int* len;  // [B]
};

__device__ __forceinline__ bool seq_ok(const PlanParams& p, const SeqArrays& s, int b, int* nq_out, int* len_out) {
  const int c0 = s.cu[b], c1 = s.cu[b + 1];
  const int len = s.len[b];
  const int nq = c1 - c0;
  *nq_out = nq;
  *len_out = len;
  return c0 >= 0 && nq >= 0 && c1 <= p.T && len >= nq && len <= p.max_seqlen_k;
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanParams p) {
  extern __shared__ int sm_plan[];
  int* cu_s = sm_plan;                // [B + 1]
  int* len_s = sm_plan + p.B + 1;     // [B]
  int* goff = len_s + p.B;            // [B + 1] group offsets of the sequences
  __shared__ int warp_sums[32];
  const int G = p.group;
  pdl_trigger();  // the indexer's prologue may start; it waits for this grid before reading the plan

  const int nt = blockDim.x;
  for (int i = threadIdx.x; i <= p.B; i += nt) {
    cu_s[i] = __ldg(p.cu_seqlens_q + i);
    if (i < p.B) len_s[i] = __ldg(p.seq_lens_k + i);
  }
  __syncthreads();
  const SeqArrays sa{cu_s, len_s};

  // (1) groups per sequence, and their offsets
  int running = 0;
  for (int b0 = 0; b0 < p.B; b0 += nt) {
    const int b = b0 + threadIdx.x;
    int ng = 0;
    if (b < p.B) {
      int nq, len;
      if (seq_ok(p, sa, b, &nq, &len)) {
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
  for (int t = threadIdx.x; t < p.T; t += nt) {
    int lo = 0, hi = p.B - 1;  // last b with cu[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu_s[mid] <= t) lo = mid; else hi = mid - 1;
    }
    int nq, len;
    const bool ok = seq_ok(p, sa, lo, &nq, &len);
    const int i = t - cu_s[lo];
    p.plan.q_seq[t] = lo;
    p.plan.q_n[t] = (ok && i >= 0 && i < nq) ? (len - nq + i + 1) / p.ratio : 0;
  }

  // (3) every group: its queries and its number of 128-key work items
  running = 0;
  for (int g0 = 0; g0 < n_groups; g0 += nt) {
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
      seq_ok(p, sa, b, &nq, &len);
      const int q0 = cu_s[b] + j * G;
      const int cnt = min(G, nq - j * G);
      const int n_last = (len - nq + j * G + cnt) / p.ratio;  // causal n (entries) of the group's last query
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
  const size_t smem = sizeof(int) * (size_t)(3 * p.B + 2);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // one thread per sequence or query up to the block's limit: a small batch
  // pays barriers and scans of a few warps, not of 32
  const int need = std::max(p.B + 1, p.T);
  const int threads = std::min(kPlanThreads, std::max(32, (need + 31) / 32 * 32));
  plan_kernel<<<1, threads, smem, stream>>>(p);
  return cudaGetLastError();
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while its predecessor on the stream still runs, and must call pdl_wait()
// before it reads anything the predecessor writes.
cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  return at;
}

}  // namespace dsa

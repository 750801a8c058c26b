// topk.cu -- exact top-k of each query's score row, ties to the lower position.
//
// "How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works / Model:
// the top-2048 past tokens are kept and a context below that is taken whole.
//
// One thread-block cluster per query row; block c of the cluster owns a
// contiguous chunk of the row.  Scores become order-preserving 32-bit keys
// (-0.0 folded onto +0.0) and a three-digit radix select (11 + 11 + 10 bits)
// finds the k-th largest key: each digit is a shared-memory histogram per
// block, summed across the cluster through distributed shared memory, so the
// row is never re-partitioned through global memory.  Each block then knows
// how many of its keys are above the threshold and how many equal it; equal
// keys are granted to the lowest positions first, and an ordered block scan
// writes the selected positions in ascending order.  When the chunk fits in
// shared memory the row is read from global memory exactly once.
#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kBins = 2048;
constexpr int kMaxCacheKeys = 45056;  // 176 KB of cached keys per block

__device__ __forceinline__ uint32_t ordered_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;  // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkParams {
  const float* scores;
  int64_t ld_scores;
  int32_t* idx;
  int64_t ld_idx;
  int32_t k;
  int32_t T;
  int32_t cache_keys;  // per-block key cache capacity (0: no cache)
  const int32_t* q_n;
  int* err;
};

// Exclusive scan of one int per thread over the block; *total gets the sum.
__device__ __forceinline__ int block_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < kThreads / 32 ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kThreads / 32) wsum[lane] = s;
  }
  __syncthreads();
  const int r = (warp ? wsum[warp - 1] : 0) + x - v;
  *total = wsum[kThreads / 32 - 1];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(TopkParams p) {
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* hist = sm;                    // [3][kBins] this block's digit histograms
  uint32_t* tot = sm + 3 * kBins;         // [kBins] cluster-summed histogram of the current digit
  uint32_t* cache = sm + 4 * kBins;       // [cache_keys]
  __shared__ int wsum[32];
  __shared__ uint32_t s_digit, s_rem, s_local_above;
  __shared__ uint32_t s_xch[2];           // this block's (keys above threshold, keys equal to it)

  const int t = blockIdx.y;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const int n = p.q_n[t];
  const int k = p.k;
  int32_t* out = p.idx + (int64_t)t * p.ld_idx;

  if (n <= k) {  // dense row (or a malformed one, n = 0): positions 0..n-1, then -1
    for (int j = crank * kThreads + threadIdx.x; j < k; j += csize * kThreads) out[j] = j < n ? j : -1;
    return;
  }

  // this block's chunk [c0, c1) of the row, 4-aligned
  const int per = ((n + csize - 1) / csize + 3) & ~3;
  const int c0 = min(n, (int)crank * per), c1 = min(n, c0 + per);
  const int len = c1 - c0;
  const bool cached = len <= p.cache_keys;
  const float* row = p.scores + (int64_t)t * p.ld_scores;

  for (int i = threadIdx.x; i < 3 * kBins; i += kThreads) hist[i] = 0;
  __syncthreads();

  uint32_t prefix = 0;   // digits fixed so far
  uint32_t rem = k;      // how many keys still to take at/below the current prefix
  uint32_t local_greater = 0;
  const int shifts[3] = {21, 10, 0};
  const uint32_t masks[3] = {0x7FFu, 0x7FFu, 0x3FFu};

  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass];
    const uint32_t msk = masks[pass];
    uint32_t* h = hist + pass * kBins;
    const int psh = sh + (pass == 0 ? 11 : (pass == 1 ? 11 : 10));  // bits above this digit
    // ---- histogram of this digit over keys matching the prefix
    if (pass == 0) {
      for (int i = threadIdx.x * 4; i < len; i += kThreads * 4) {
        const int s = c0 + i;
        float v[4];
        if (s + 3 < c1) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(row + s));
          v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        } else {
          for (int j = 0; j < 4; ++j) v[j] = (s + j < c1) ? row[s + j] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (s + j >= c1) break;
          const uint32_t key = ordered_key(v[j]);
          if (cached) cache[i + j] = key;
          atomicAdd(&h[key >> sh], 1u);
        }
      }
    } else {
      for (int i = threadIdx.x; i < len; i += kThreads) {
        const uint32_t key = cached ? cache[i] : ordered_key(row[c0 + i]);
        if ((key >> psh) == prefix) atomicAdd(&h[(key >> sh) & msk], 1u);
      }
    }
    cluster_sync();  // every block's histogram of this digit is complete
    // ---- cluster-wide histogram
    for (int bin = threadIdx.x; bin < kBins; bin += kThreads) {
      uint32_t sum = 0;
      const uint32_t local = smem_u32(h + bin);
      for (uint32_t r = 0; r < csize; ++r) sum += (r == crank) ? h[bin] : ld_dsmem_u32(dsmem_addr(local, r));
      tot[bin] = sum;
    }
    __syncthreads();
    // ---- the digit holding the rem-th largest key: suffix sums from the top bin
    {
      const int nb = (int)msk + 1;        // bins of this digit
      const int per_t = (nb + kThreads - 1) / kThreads;  // 4 or 2
      const int hi = nb - 1 - threadIdx.x * per_t;       // this thread's bins: hi, hi-1, ...
      int mine = 0;
      for (int j = 0; j < per_t; ++j) if (hi - j >= 0) mine += tot[hi - j];
      int total;
      int above = block_scan(mine, wsum, &total);        // keys in bins above this thread's
      for (int j = 0; j < per_t; ++j) {
        const int bin = hi - j;
        if (bin < 0) break;
        const int c = tot[bin];
        if ((uint32_t)above < rem && rem <= (uint32_t)(above + c)) {
          s_digit = bin;
          s_rem = rem - above;
        }
        above += c;
      }
      if (threadIdx.x == 0) s_local_above = 0;
      __syncthreads();
      const uint32_t d = s_digit;
      // this block's own keys in bins above the chosen digit
      uint32_t la = 0;
      for (int bin = d + 1 + threadIdx.x; bin < nb; bin += kThreads) la += h[bin];
      if (la) atomicAdd(&s_local_above, la);
      __syncthreads();
      local_greater += s_local_above;
      prefix = (prefix << (psh - sh)) | d;
      rem = s_rem;
      __syncthreads();
    }
  }
  const uint32_t thr = prefix;  // the k-th largest key
  const uint32_t local_equal = hist[2 * kBins + (thr & 0x3FFu)];
  if (threadIdx.x == 0) {
    s_xch[0] = local_greater;
    s_xch[1] = local_equal;
  }
  cluster_sync();
  // output offset of this block and the number of equal keys it may take
  uint32_t base = 0, eq_before = 0;
  for (uint32_t r = 0; r < crank; ++r) {
    const uint32_t g = ld_dsmem_u32(dsmem_addr(smem_u32(&s_xch[0]), r));
    const uint32_t e = ld_dsmem_u32(dsmem_addr(smem_u32(&s_xch[1]), r));
    const uint32_t take_r = min(e, rem > eq_before ? rem - eq_before : 0u);
    base += g + take_r;
    eq_before += e;
  }
  const uint32_t take = min(local_equal, rem > eq_before ? rem - eq_before : 0u);

  // ordered compaction: positions in ascending order
  uint32_t eq_run = 0, sel_run = 0;
  for (int i0 = 0; i0 < len; i0 += kThreads * 4) {
    const int i = i0 + threadIdx.x * 4;
    uint32_t key[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (i + j < len) key[j] = cached ? cache[i + j] : ordered_key(row[c0 + i + j]);
      else key[j] = 0u;  // below every real key
    }
    int n_eq = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) n_eq += (i + j < len && key[j] == thr);
    int eq_tot;
    int eq_rank = (int)eq_run + block_scan(n_eq, wsum, &eq_tot);
    bool sel[4];
    int n_sel = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool valid = i + j < len;
      const bool eq = valid && key[j] == thr;
      sel[j] = valid && (key[j] > thr || (eq && (uint32_t)eq_rank < take));
      if (eq) ++eq_rank;
      n_sel += sel[j];
    }
    int sel_tot;
    int pos = (int)(base + sel_run) + block_scan(n_sel, wsum, &sel_tot);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (sel[j]) {
        if (pos < k) out[pos] = c0 + i + j;
        ++pos;
      }
    eq_run += eq_tot;
    sel_run += sel_tot;
  }
  cluster_sync();  // peers may still read this block's shared memory
}

int g_max_cluster = 0;  // largest cluster size the device schedules for this kernel

}  // namespace

cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  // cluster size: enough blocks to fill the GPU on few rows, and chunks that
  // fit the shared-memory key cache when possible
  int c = 1;
  while (c < 16 && (int64_t)a.T * c * 2 <= a.num_sms) c *= 2;
  while (c < 16 && (a.max_n + c - 1) / c > kMaxCacheKeys) c *= 2;
  if (g_max_cluster == 0) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    g_max_cluster = 8;
    cudaLaunchConfig_t probe = {};
    probe.gridDim = dim3(16, 1, 1);
    probe.blockDim = dim3(kThreads, 1, 1);
    probe.dynamicSmemBytes = (4 * kBins + kMaxCacheKeys) * 4;
    e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)probe.dynamicSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 16;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    probe.attrs = &at;
    probe.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, topk_kernel, &probe) == cudaSuccess && nclusters > 0)
      g_max_cluster = 16;
    cudaGetLastError();
  }
  if (c > g_max_cluster) c = g_max_cluster;
  const int per = (((a.max_n + c - 1) / c) + 3) & ~3;
  const int cache_keys = per <= kMaxCacheKeys ? per : 0;
  const size_t smem = (size_t)(4 * kBins + cache_keys) * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;

  TopkParams p;
  p.scores = a.scores;
  p.ld_scores = a.ld_scores;
  p.idx = a.idx;
  p.ld_idx = a.ld_idx;
  p.k = a.k;
  p.T = a.T;
  p.cache_keys = cache_keys;
  p.q_n = a.q_n;
  p.err = a.err;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c, a.T, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = c;
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel, p);
}

}  // namespace dsa

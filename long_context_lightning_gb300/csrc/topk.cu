// topk.cu -- exact top-k of each query's score row, ties to the lower position.
//
// "How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works / Model:
// the top-2048 past tokens are kept and a context below that is taken whole.
//
// One thread-block cluster per query row (one block when the row fits); block
// c of the cluster owns a contiguous chunk of the row.  Scores become
// order-preserving 32-bit keys (-0.0 folded onto +0.0) and a three-digit radix
// select (11 + 11 + 10 bits) finds the k-th largest key: each digit is a
// shared-memory histogram per block, summed across the cluster through
// distributed shared memory.  Each block then knows how many of its keys are
// above the threshold and how many equal it; equal keys are granted to the
// lowest positions first.  The ordered write is per thread: each thread owns
// a contiguous run of the chunk and places its selections after one block scan
// of the threads' counts.  When the chunk fits in shared memory the row is read
// from global memory exactly once.
//
// Candidate path (taken when it fits, decided the same way by every block):
// after the first digit, the keys at or above its bin -- the k selections plus
// the rest of the threshold bin, usually a few hundred more -- are few.  Every
// block sends its candidates, in position order, into the shared memory of
// the cluster's first block (one atomic reserves a contiguous segment, a table
// records it by block rank); after one more cluster barrier that block alone
// finishes the last two digits over the candidates and writes the row in
// position order.  Two cluster barriers instead of four, and the last two
// digits touch only the candidates.
#include <algorithm>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kMaxCacheKeys = 32768;  // 128 KB of cached keys per block
constexpr int kCand = 8192;           // candidate capacity of the first block (64 KB of (key, position))
constexpr int kMaxCluster = 16;

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
  int32_t plan_early;  // the plan was written two or more grids back
  int32_t cand;        // the first block has room for the candidate path
};

__device__ __forceinline__ int warp_excl_scan(int v) {
  const int lane = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x - v;
}

__device__ __forceinline__ void hist_add(uint32_t* h, uint32_t bin, bool active) {
  if (active) atomicAdd(&h[bin], 1u);
}

// Block-wide exclusive scan of one int per thread (kThreads threads); returns
// the prefix and the total.  Uses a[kWarps] and b[kWarps] as scratch.
__device__ __forceinline__ int block_scan(int v, int* a, int* b, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ex = warp_excl_scan(v);
  if (lane == 31) a[warp] = ex + v;
  __syncthreads();
  if (warp == 0) b[lane] = warp_excl_scan(a[lane]);
  __syncthreads();
  const int r = b[warp] + ex;
  *total = b[kWarps - 1] + a[kWarps - 1];
  __syncthreads();
  return r;
}

// One block: the digit (over bins [0, nb) of histogram h) that holds the
// rem-th largest key, and the rank left inside it.
__device__ __forceinline__ void block_select_digit(const uint32_t* h, int nb, uint32_t rem, int* a, int* b,
                                                   uint32_t* s_digit, uint32_t* s_rem) {
  const int bpt = nb / kThreads;
  const int top = nb - 1 - (int)threadIdx.x * bpt;
  int mine = 0;
  for (int j = 0; j < bpt; ++j) mine += (int)h[top - j];
  int total;
  int acc = block_scan(mine, a, b, &total);
  if ((uint32_t)acc < rem && rem <= (uint32_t)(acc + mine)) {
    for (int j = 0; j < bpt; ++j) {
      const int cnt = (int)h[top - j];
      if ((uint32_t)(acc + cnt) >= rem) {
        *s_digit = top - j;
        *s_rem = rem - acc;
        break;
      }
      acc += cnt;
    }
  }
  __syncthreads();
}

template <class Keys4>
__device__ __forceinline__ void candidate_path(const TopkParams& p, uint32_t* hist, uint2* cand, bool cached, Keys4 keys4,
                                            int len, int c0, uint32_t d0, uint32_t rem0, uint32_t own_above,
                                            uint32_t crank, uint32_t csize, int32_t* out, int* w_a, int* w_b,
                                            int* w_c, int* w_d, uint32_t* s_cand_n, uint32_t (*s_seg)[2],
                                            uint32_t* s_cbase, uint32_t* s_digit, uint32_t* s_rem) {
  (void)cached;
  const int k = p.k;
  // (1) this block's candidates: its keys whose first digit is d0 or above, in position order
  const uint32_t mine = own_above + hist[d0];
  if (threadIdx.x == 0) {
    const uint32_t base = atom_add_dsmem_u32(dsmem_addr(smem_u32(s_cand_n), 0), mine);
    *s_cbase = base;
    st_dsmem_u32(dsmem_addr(smem_u32(&s_seg[crank][0]), 0), base);
    st_dsmem_u32(dsmem_addr(smem_u32(&s_seg[crank][1]), 0), mine);
  }
  const int R = ((len + kThreads - 1) / kThreads + 3) & ~3;
  const int r0 = min(len, (int)threadIdx.x * R), r1 = min(len, r0 + R);
  int cnt = 0;
  for (int i = r0; i < r1; i += 4) {
    uint32_t kk[4];
    keys4(i, kk);
#pragma unroll
    for (int j = 0; j < 4; ++j) cnt += (i + j < r1) && (kk[j] >> 21) >= d0;
  }
  int total;
  const int before = block_scan(cnt, w_a, w_b, &total);  // also orders s_cbase before its use
  uint32_t slot = *s_cbase + (uint32_t)before;
  const uint32_t cand0 = dsmem_addr(smem_u32(cand), 0);
  for (int i = r0; i < r1; i += 4) {
    uint32_t kk[4];
    keys4(i, kk);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if ((i + j < r1) && (kk[j] >> 21) >= d0) {
        st_dsmem_v2_u32(cand0 + slot * 8u, kk[j], (uint32_t)(c0 + i + j));
        ++slot;
      }
  }
  cluster_sync();  // every block's candidates are in the first block; no one reads a peer's memory after this
  if (crank != 0) return;

  // (2) the first block: the last two digits among the candidates of bin d0
  const int n_c = (int)*s_cand_n;
  uint32_t* h1 = hist + kBins;
  uint32_t* h2 = hist + 2 * kBins;
  for (int i = threadIdx.x; i < n_c; i += kThreads) {
    const uint32_t key = cand[i].x;
    if ((key >> 21) == d0) atomicAdd(&h1[(key >> 10) & 0x7FFu], 1u);
  }
  __syncthreads();
  block_select_digit(h1, kBins, rem0, w_a, w_b, s_digit, s_rem);
  const uint32_t d1 = *s_digit, rem1 = *s_rem;
  const uint32_t pre = (d0 << 11) | d1;
  for (int i = threadIdx.x; i < n_c; i += kThreads) {
    const uint32_t key = cand[i].x;
    if ((key >> 10) == pre) atomicAdd(&h2[key & 0x3FFu], 1u);
  }
  __syncthreads();
  block_select_digit(h2, 1024, rem1, w_a, w_b, s_digit, s_rem);
  const uint32_t thr = (pre << 10) | *s_digit;  // the k-th largest key
  const int take = (int)*s_rem;                 // keys equal to it that are selected (lowest positions first)

  // (3) ordered write: segments in block-rank order, each in position order
  int out_pos = 0, eq_taken = 0;
  for (uint32_t r = 0; r < csize; ++r) {
    const int sb = (int)s_seg[r][0], sc = (int)s_seg[r][1];
    const int Rs = (sc + kThreads - 1) / kThreads;
    const int a0 = min(sc, (int)threadIdx.x * Rs), a1 = min(sc, a0 + Rs);
    int gt = 0, eq = 0;
    for (int i = a0; i < a1; ++i) {
      const uint32_t key = cand[sb + i].x;
      gt += key > thr;
      eq += key == thr;
    }
    int gt_tot, eq_tot;
    const int gt_before = block_scan(gt, w_a, w_b, &gt_tot);
    const int eq_before = block_scan(eq, w_c, w_d, &eq_tot);
    const int left = take - eq_taken;
    const int allow = max(0, min(eq, left - eq_before));
    int pos = out_pos + gt_before + min(eq_before, max(left, 0));
    int eq_seen = 0;
    for (int i = a0; i < a1; ++i) {
      const uint2 c = cand[sb + i];
      const bool e = c.x == thr;
      if (c.x > thr || (e && eq_seen < allow)) {
        if (pos < k) out[pos] = (int32_t)c.y;
        ++pos;
      }
      eq_seen += e;
    }
    const int eq_used = min(eq_tot, max(left, 0));
    out_pos += gt_tot + eq_used;
    eq_taken += eq_used;
  }
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(TopkParams p) {
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* hist = sm;                    // [3][kBins] this block's digit histograms
  uint32_t* tot = sm + 3 * kBins;         // [kBins] cluster-summed histogram of the current digit
  uint32_t* cache = sm + 4 * kBins;       // [cache_keys]
  uint2* cand = reinterpret_cast<uint2*>(cache + p.cache_keys);  // [kCand] (key, position), first block only
  __shared__ int w_gt[kWarps], w_eq[kWarps], w_eqb[kWarps], w_selb[kWarps];
  __shared__ uint32_t s_digit, s_rem, s_local_above;
  __shared__ uint32_t s_xch[2];           // this block's (keys above threshold, keys equal to it)
  __shared__ uint32_t s_cand_n;           // first block: candidate slots reserved so far
  __shared__ uint32_t s_seg[kMaxCluster][2];  // first block: (first slot, count) of each block's candidates
  __shared__ uint32_t s_cbase;

  const int t = blockIdx.y;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  int n = p.plan_early ? __ldcg(p.q_n + t) : 0;
  pdl_wait();  // scores and plan of the previous grids are complete from here on
  pdl_trigger();
  if (!p.plan_early) n = p.q_n[t];
  const int k = p.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
  if (threadIdx.x == 0) s_cand_n = 0;  // before the first cluster barrier, so before any peer's reservation
  __syncthreads();
  auto keys4 = [&](int i, uint32_t* kk) {  // keys i..i+3 of the chunk (i a multiple of 4, i < len)
    if (cached) {
      const uint4 q = *reinterpret_cast<const uint4*>(cache + i);  // within the cache: len <= its 4-aligned size
      kk[0] = q.x; kk[1] = q.y; kk[2] = q.z; kk[3] = q.w;
    } else if (c0 + i + 3 < c1) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row + c0 + i));
      kk[0] = ordered_key(f.x); kk[1] = ordered_key(f.y); kk[2] = ordered_key(f.z); kk[3] = ordered_key(f.w);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) kk[j] = (c0 + i + j < c1) ? ordered_key(row[c0 + i + j]) : 0u;
    }
  };

  uint32_t prefix = 0;   // digits fixed so far
  uint32_t rem = k;      // how many keys still to take at/below the current prefix
  uint32_t local_greater = 0;

#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int bits = pass == 2 ? 10 : 11;
    const uint32_t msk = (1u << bits) - 1u;
    const int psh = sh + bits;  // bits above this digit
    uint32_t* h = hist + pass * kBins;
    // ---- histogram of this digit over keys matching the prefix
    if (pass == 0) {
      // four 16-byte loads in flight per thread before any is used
      for (int i0 = 0; i0 < len; i0 += kThreads * 16) {
        float v[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + (u * kThreads + (int)threadIdx.x) * 4;
          const int s = c0 + i;
          if (s + 3 < c1) {
            const float4 f = __ldg(reinterpret_cast<const float4*>(row + s));
            v[4 * u] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[4 * u + j] = (s + j < c1) ? row[s + j] : 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + (u * kThreads + (int)threadIdx.x) * 4;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const bool in = c0 + i + j < c1;
            const uint32_t key = ordered_key(v[4 * u + j]);
            if (cached && in) cache[i + j] = key;
            hist_add(h, key >> sh, in);
          }
        }
      }
    } else {
      for (int i = (int)threadIdx.x * 4; i < len; i += kThreads * 4) {  // four keys per step
        uint32_t kk[4];
        keys4(i, kk);
#pragma unroll
        for (int j = 0; j < 4; ++j) hist_add(h, (kk[j] >> sh) & msk, i + j < len && (kk[j] >> psh) == prefix);
      }
    }
    cluster_sync();  // every block's histogram of this digit is complete
    // ---- cluster-wide histogram and the digit holding the rem-th largest key.
    // Thread t owns the bins just below those of thread t-1 (thread 0 the top
    // ones); it sums them over the cluster, and one block scan of (cluster
    // count, own count) pairs gives, at the chosen digit, both the keys above
    // it in the cluster and this block's own keys above it.
    const int nb = (int)msk + 1;
    const int bpt = nb / kThreads;  // 2 or 1 bins per thread
    const int top = nb - 1 - (int)threadIdx.x * bpt;
    int tot_mine = 0, own_mine = 0;
    if (bpt == 2) {
      // the thread's two bins are adjacent and 8-byte aligned: one remote load per peer
      const int b0 = top - 1;
      uint32_t s0 = h[b0], s1 = h[b0 + 1];
      const uint32_t local = smem_u32(h + b0);
      for (uint32_t r = 0; r < csize; ++r)
        if (r != crank) {
          const uint2 v = ld_dsmem_v2_u32(dsmem_addr(local, r));
          s0 += v.x;
          s1 += v.y;
        }
      tot[b0] = s0;
      tot[b0 + 1] = s1;
      tot_mine = (int)(s0 + s1);
      own_mine = (int)(h[b0] + h[b0 + 1]);
    } else {
      uint32_t sum = h[top];
      const uint32_t local = smem_u32(h + top);
      for (uint32_t r = 0; r < csize; ++r)
        if (r != crank) sum += ld_dsmem_u32(dsmem_addr(local, r));
      tot[top] = sum;
      tot_mine = (int)sum;
      own_mine = (int)h[top];
    }
    const int tot_ex = warp_excl_scan(tot_mine), own_ex = warp_excl_scan(own_mine);
    if (lane == 31) {
      w_gt[warp] = tot_ex + tot_mine;  // warp totals (reusing the write-phase scratch)
      w_eq[warp] = own_ex + own_mine;
    }
    __syncthreads();
    if (warp == 0) {
      const int a_t = w_gt[lane], a_o = w_eq[lane];
      w_eqb[lane] = warp_excl_scan(a_t);
      w_selb[lane] = warp_excl_scan(a_o);
    }
    __syncthreads();
    {
      int acc_t = w_eqb[warp] + tot_ex, acc_o = w_selb[warp] + own_ex;  // keys above this thread's bins
      if ((uint32_t)acc_t < rem && rem <= (uint32_t)(acc_t + tot_mine)) {
        for (int j = 0; j < bpt; ++j) {
          const int bin = top - j;
          const int cnt = (int)tot[bin];
          if ((uint32_t)(acc_t + cnt) >= rem) {
            s_digit = bin;
            s_rem = rem - acc_t;
            s_local_above = acc_o;
            break;
          }
          acc_t += cnt;
          acc_o += (int)h[bin];
        }
      }
    }
    __syncthreads();
    local_greater += s_local_above;
    prefix = (prefix << bits) | s_digit;
    rem = s_rem;
    if (pass == 0 && p.cand && (uint32_t)k - rem + tot[prefix] <= (uint32_t)kCand) {
      candidate_path(p, hist, cand, cached, keys4, len, c0, prefix, rem, local_greater, crank, csize, out, w_gt,
                     w_eq, w_selb, w_eqb, &s_cand_n, s_seg, &s_cbase, &s_digit, &s_rem);
      return;
    }
    __syncthreads();  // the next pass rewrites s_digit, s_rem, s_local_above and the scratch
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
  const int take = (int)min(local_equal, rem > eq_before ? rem - eq_before : 0u);
  // the last remote reads are done: a block may leave once every peer has
  // also passed this point (the wait is at the end)
  cluster_arrive();

  // ---- ordered write: thread t owns the contiguous run [t*R, t*R + R) of the
  // chunk (R a multiple of four, so keys are read four at a time).  A counting
  // pass records which of its keys are above / equal to the threshold as bits
  // (runs up to 64 keys), one block scan of the two counts places every
  // thread's first selection, and each thread writes its own selections in
  // position order.  Equal keys go to the lowest positions: those a thread
  // may take are what is left of the block's allowance after the threads
  // before it.
  const int R = ((len + kThreads - 1) / kThreads + 3) & ~3;
  const int r0 = min(len, (int)threadIdx.x * R), r1 = min(len, r0 + R);
  const bool in_regs = R <= 64;
  uint64_t gtb = 0, eqb = 0;
  int gt = 0, eq = 0;
  for (int i = r0; i < r1; i += 4) {
    uint32_t kk[4];
    keys4(i, kk);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool in = i + j < r1;
      const bool g = in && kk[j] > thr, e = in && kk[j] == thr;
      gt += g;
      eq += e;
      if (in_regs) {
        gtb |= (uint64_t)g << (i - r0 + j);
        eqb |= (uint64_t)e << (i - r0 + j);
      }
    }
  }
  // block-exclusive scans of (above, equal) counts: lanes, then warps
  const int gt_ex = warp_excl_scan(gt), eq_ex = warp_excl_scan(eq);
  if (lane == 31) {
    w_gt[warp] = gt_ex + gt;
    w_eq[warp] = eq_ex + eq;
  }
  __syncthreads();
  if (warp == 0) {
    w_selb[lane] = warp_excl_scan(w_gt[lane]);
    w_eqb[lane] = warp_excl_scan(w_eq[lane]);
  }
  __syncthreads();
  {
    const int gt_before = w_selb[warp] + gt_ex, eq_before_t = w_eqb[warp] + eq_ex;
    const int allow = max(0, min(eq, take - eq_before_t));  // this thread's equal keys that are taken
    int pos = (int)base + gt_before + min(eq_before_t, take);
    if (in_regs) {
      // the first `allow` equal keys, then every selection in position order
      uint64_t eqa = 0, em = eqb;
      for (int a = 0; a < allow; ++a) {
        const uint64_t low = em & (~em + 1);
        eqa |= low;
        em ^= low;
      }
      uint64_t sel = gtb | eqa;
      while (sel) {
        const int j = __ffsll((long long)sel) - 1;
        sel &= sel - 1;
        if (pos < k) out[pos] = c0 + r0 + j;
        ++pos;
      }
    } else {
      int eq_seen = 0;
      for (int i = r0; i < r1; i += 4) {
        uint32_t kk[4];
        keys4(i, kk);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (i + j >= r1) continue;
          const bool e = kk[j] == thr;
          if (kk[j] > thr || (e && eq_seen < allow)) {
            if (pos < k) out[pos] = c0 + i + j;
            ++pos;
          }
          eq_seen += e;
        }
      }
    }
  }
  cluster_wait();  // peers may still read this block's shared memory until they arrive
}

}  // namespace

cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const int probe_smem = (4 * kBins + kMaxCacheKeys + 2 * kCand) * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, probe_smem);
  if (e != cudaSuccess) return e;
  int max_cluster = max_cluster_for(reinterpret_cast<const void*>(topk_kernel), kThreads, probe_smem,
                                    kClusterSlotTopk);
  if (max_cluster == 0) return cudaErrorUnknown;
  if (topk_cluster_cap() > 0) max_cluster = std::min(max_cluster, topk_cluster_cap());
  // cluster size: enough blocks per row that the rows fill a good share of the
  // GPU (each block reads less of the row), and chunks that fit the key cache
  int c = 1;
  while (c < max_cluster && (a.max_n + c - 1) / c > kMaxCacheKeys) c *= 2;
  while (c < max_cluster && (int64_t)a.T * c * 2 <= a.num_sms && (a.max_n + 2 * c - 1) / (2 * c) >= 4096) c *= 2;
  const int per = (((a.max_n + c - 1) / c) + 3) & ~3;
  const int cache_keys = per <= kMaxCacheKeys ? per : 0;
  const size_t smem = (size_t)(4 * kBins + cache_keys + 2 * kCand) * 4;
  e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  p.plan_early = a.plan_early ? 1 : 0;
  p.cand = (c <= kMaxCluster && !topk_three_pass_only()) ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c, a.T, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = c;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1] = pdl_attribute();
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, topk_kernel, p);
}

}  // namespace dsa

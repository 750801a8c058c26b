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
  int32_t cache_half;  // the cache holds the top 16 bits of each key (chunks up to twice as long)
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
__device__ __forceinline__ void candidate_path(const TopkParams& p, uint32_t* hist, uint2* cand, bool cached, bool half,
                                               const uint16_t* cache16, Keys4 keys4,
                                            int len, int c0, uint32_t d0, uint32_t rem0, uint32_t own_above,
                                            uint32_t crank, uint32_t csize, int32_t* out, int* w_a, int* w_b,
                                            int* w_c, int* w_d, uint32_t* s_cand_n, uint32_t (*s_seg)[2],
                                            uint32_t* s_cbase, uint32_t* s_digit, uint32_t* s_rem) {
  const int k = p.k;
  // (1) this block's candidates: its keys whose first digit is d0 or above, in position order
  const uint32_t mine = own_above + hist[d0];
  if (threadIdx.x == 0) {
    const uint32_t base = atom_add_dsmem_u32(dsmem_addr(smem_u32(s_cand_n), 0), mine);
    *s_cbase = base;
    st_dsmem_u32(dsmem_addr(smem_u32(&s_seg[crank][0]), 0), base);
    st_dsmem_u32(dsmem_addr(smem_u32(&s_seg[crank][1]), 0), mine);
  }
  const uint32_t cand0 = dsmem_addr(smem_u32(cand), 0);
  if (cached) {
    // thread t owns a contiguous run of the cached chunk
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
  } else if (half) {
    // thread t owns a contiguous run of the cached key tops (eight per
    // 16-byte read); a candidate's full key is read back from global memory
    const float* row = p.scores + (int64_t)blockIdx.y * p.ld_scores;
    const int R = ((len + kThreads - 1) / kThreads + 7) & ~7;
    const int r0 = min(len, (int)threadIdx.x * R), r1 = min(len, r0 + R);
    int cnt = 0;
    for (int i = r0; i < r1; i += 8) {
      const uint4 q = *reinterpret_cast<const uint4*>(cache16 + i);
      const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) cnt += (i + j < r1) && (((w4[j >> 1] >> (16 * (j & 1))) & 0xFFFFu) >> 5) >= d0;
    }
    int total;
    const int before = block_scan(cnt, w_a, w_b, &total);  // also orders s_cbase before its use
    uint32_t slot = *s_cbase + (uint32_t)before;
    for (int i = r0; i < r1; i += 8) {
      const uint4 q = *reinterpret_cast<const uint4*>(cache16 + i);
      const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
      uint32_t cm = 0;  // which of the eight are candidates
#pragma unroll
      for (int j = 0; j < 8; ++j)
        cm |= (uint32_t)((i + j < r1) && (((w4[j >> 1] >> (16 * (j & 1))) & 0xFFFFu) >> 5) >= d0) << j;
      if (cm) {
        float f[8];  // the candidates' full scores, loads in flight together
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = ((cm >> j) & 1u) ? row[c0 + i + j] : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if ((cm >> j) & 1u) {
            st_dsmem_v2_u32(cand0 + slot * 8u, ordered_key(f[j]), (uint32_t)(c0 + i + j));
            ++slot;
          }
      }
    }
  } else {
    // the chunk is read from global memory: warp w owns the contiguous span
    // [w S, w S + S) (S a multiple of 512), read 512 keys at a time (four
    // 16-byte loads in flight per lane); a counting pass, one scan of the warps'
    // counts, then a writing pass that places each 128-key step with a warp scan
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int S = ((len + kWarps * 512 - 1) / (kWarps * 512)) * 512;
    const int s0 = min(len, warp * S), s1 = min(len, s0 + S);
    auto load4 = [&](int i, uint32_t* kk) {  // keys i..i+3 of the chunk (i a multiple of 4), 0 past the span
      if (i + 3 < s1) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p.scores + (int64_t)blockIdx.y * p.ld_scores + c0 + i));
        kk[0] = ordered_key(f.x); kk[1] = ordered_key(f.y); kk[2] = ordered_key(f.z); kk[3] = ordered_key(f.w);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          kk[j] = (i + j < s1) ? ordered_key(p.scores[(int64_t)blockIdx.y * p.ld_scores + c0 + i + j]) : 0u;
      }
    };
    int cnt = 0;
    for (int i0 = s0; i0 < s1; i0 += 512) {
      uint32_t kk[16];
#pragma unroll
      for (int u = 0; u < 4; ++u) load4(i0 + u * 128 + lane * 4, kk + 4 * u);
#pragma unroll
      for (int u = 0; u < 16; ++u) cnt += (i0 + (u >> 2) * 128 + lane * 4 + (u & 3) < s1) && (kk[u] >> 21) >= d0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    int total;
    const int before = block_scan(lane == 0 ? cnt : 0, w_a, w_b, &total);  // lane 0 carries its warp's count
    uint32_t slot = *s_cbase + (uint32_t)__shfl_sync(0xffffffffu, before, 0);
    for (int i0 = s0; i0 < s1; i0 += 512) {
      uint32_t kk[16];
#pragma unroll
      for (int u = 0; u < 4; ++u) load4(i0 + u * 128 + lane * 4, kk + 4 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * 128 + lane * 4;
        int c = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) c += (i + j < s1) && (kk[4 * u + j] >> 21) >= d0;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        uint32_t q = slot + (uint32_t)(incl - c);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if ((i + j < s1) && (kk[4 * u + j] >> 21) >= d0) {
            st_dsmem_v2_u32(cand0 + q * 8u, kk[4 * u + j], (uint32_t)(c0 + i + j));
            ++q;
          }
        slot += (uint32_t)__shfl_sync(0xffffffffu, incl, 31);
      }
    }
  }
  cluster_sync();  // every block's candidates are in the first block; no one reads a peer's memory after this
  if (crank != 0) return;

  // (2) the first block: the last two digits among the candidates of bin d0
  __shared__ uint32_t s_lo[kMaxCluster + 1];  // logical start of each block's segment (block-rank order)
  if (threadIdx.x == 0) {
    s_lo[0] = 0;
    for (int r = 0; r < kMaxCluster; ++r) s_lo[r + 1] = s_lo[r] + ((uint32_t)r < csize ? s_seg[r][1] : 0u);
  }
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

  // (3) ordered write in one pass.  Logical candidate order = the segments in
  // block-rank order, each in position order; thread t owns a contiguous run
  // of it.  One scan of packed (above, equal) counts (both < 2^16) places
  // every thread's first selection; equal keys go to the lowest positions.
  auto phys = [&](int L, int& r) {  // physical slot of logical index L; r is the segment, advanced as L grows
    while ((uint32_t)L >= s_lo[r + 1]) ++r;
    return (int)s_seg[r][0] + L - (int)s_lo[r];
  };
  const int Rs = (n_c + kThreads - 1) / kThreads;
  const int a0 = min(n_c, (int)threadIdx.x * Rs), a1 = min(n_c, a0 + Rs);
  int gt = 0, eq = 0;
  {
    int r = 0;
    for (int L = a0; L < a1; ++L) {
      const uint32_t key = cand[phys(L, r)].x;
      gt += key > thr;
      eq += key == thr;
    }
  }
  int packed_tot;
  const int packed_before = block_scan(gt | (eq << 16), w_a, w_b, &packed_tot);
  const int gt_before = packed_before & 0xFFFF, eq_before = packed_before >> 16;
  const int allow = max(0, min(eq, take - eq_before));
  int pos = gt_before + min(eq_before, take);
  {
    int r = 0, eq_seen = 0;
    for (int L = a0; L < a1; ++L) {
      const uint2 c = cand[phys(L, r)];
      const bool e = c.x == thr;
      if (c.x > thr || (e && eq_seen < allow)) {
        if (pos < k) out[pos] = (int32_t)c.y;
        ++pos;
      }
      eq_seen += e;
    }
  }
  (void)w_c;
  (void)w_d;
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(TopkParams p) {
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* hist = sm;                    // [3][kBins] this block's digit histograms
  uint32_t* cache = sm + 3 * kBins;       // [cache_keys] keys, or [cache_keys] 16-bit key tops
  uint16_t* cache16 = reinterpret_cast<uint16_t*>(cache);
  uint2* cand = reinterpret_cast<uint2*>(cache + (p.cache_half ? p.cache_keys / 2 : p.cache_keys));  // [kCand]
  __shared__ int w_gt[kWarps], w_eq[kWarps], w_eqb[kWarps], w_selb[kWarps];
  __shared__ uint32_t s_digit, s_rem, s_local_above;
  __shared__ uint32_t s_xch[2];           // this block's (keys above threshold, keys equal to it)
  __shared__ uint32_t s_cand_n;           // first block: candidate slots reserved so far
  __shared__ uint32_t s_seg[kMaxCluster][2];  // first block: (first slot, count) of each block's candidates
  __shared__ uint32_t s_cbase;
  __shared__ uint32_t coarse[3][64];      // per digit: this block's sums of 32 consecutive bins
  __shared__ uint32_t s_tot_d;            // the cluster's count of the chosen digit's bin

  const int t = blockIdx.y;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  // block-local set-up needs nothing from the previous grids: done before waiting for them
  for (int i = threadIdx.x; i < 3 * kBins; i += kThreads) hist[i] = 0;
  if (threadIdx.x == 0) s_cand_n = 0;  // before the first cluster barrier, so before any peer's reservation
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
  const bool cached = !p.cache_half && len <= p.cache_keys;
  const bool half = p.cache_half && len <= p.cache_keys;
  const float* row = p.scores + (int64_t)t * p.ld_scores;

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
            if (half && in) cache16[i + j] = (uint16_t)(key >> 16);
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
    // ---- coarse sums of this block's histogram: group g = bins [32 g, 32 g + 32)
    const int nb = (int)msk + 1;
    const int ng = nb / 32;  // 64 or 32 groups
    __syncthreads();         // every thread's histogram adds are done
    for (int g = warp; g < ng; g += kWarps) {
      uint32_t v = h[g * 32 + lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) coarse[pass][g] = v;
    }
    cluster_sync();  // every block's histogram and coarse sums of this digit are complete
    // ---- the digit holding the rem-th largest key (warp 0): the cluster's
    // coarse sums, top group first, pick a group; the cluster's counts of its 32
    // bins pick the digit.  Exclusive scans of the cluster counts and of this
    // block's own counts give, at the pick, the keys above it in the cluster
    // and this block's own keys above it.
    if (warp == 0) {
      auto peer_sum = [&](const uint32_t* v) -> uint32_t {  // over the other blocks, four loads in flight
        const uint32_t local = smem_u32(v);
        uint32_t sum = 0;
        for (uint32_t rb = 0; rb < csize; rb += 4) {
          uint32_t x[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t r = rb + j;
            x[j] = (r < csize && r != crank) ? ld_dsmem_u32(dsmem_addr(local, r)) : 0u;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) sum += x[j];
        }
        return sum;
      };
      const int gpl = ng / 32;  // groups per lane, lane 0 the top ones
      uint32_t c_all[2] = {0u, 0u}, c_own[2] = {0u, 0u};
      for (int j = 0; j < gpl; ++j) {
        const int g = ng - 1 - lane * gpl - j;
        c_own[j] = coarse[pass][g];
        c_all[j] = c_own[j] + peer_sum(&coarse[pass][g]);
      }
      const uint32_t lane_all = c_all[0] + c_all[1], lane_own = c_own[0] + c_own[1];
      const uint32_t ex_all = (uint32_t)warp_excl_scan((int)lane_all), ex_own = (uint32_t)warp_excl_scan((int)lane_own);
      const unsigned m = __ballot_sync(0xffffffffu, ex_all < rem && rem <= ex_all + lane_all);
      const int src = m ? __ffs(m) - 1 : 31;
      int G = 0;
      uint32_t above_all = 0, above_own = 0;
      if (lane == src) {
        uint32_t acc = ex_all, acco = ex_own;
        for (int j = 0; j < gpl; ++j) {
          G = ng - 1 - lane * gpl - j;
          if (acc + c_all[j] >= rem) break;
          acc += c_all[j];
          acco += c_own[j];
        }
        above_all = acc;
        above_own = acco;
      }
      G = __shfl_sync(0xffffffffu, G, src);
      above_all = __shfl_sync(0xffffffffu, above_all, src);
      above_own = __shfl_sync(0xffffffffu, above_own, src);
      const uint32_t rem_g = rem - above_all;
      const int b = G * 32 + 31 - lane;  // lane 0 the group's top bin
      const uint32_t f_own = h[b], f_all = f_own + peer_sum(&h[b]);
      const uint32_t fx_all = (uint32_t)warp_excl_scan((int)f_all), fx_own = (uint32_t)warp_excl_scan((int)f_own);
      const unsigned fm = __ballot_sync(0xffffffffu, fx_all < rem_g && rem_g <= fx_all + f_all);
      if (lane == (fm ? __ffs(fm) - 1 : 31)) {
        s_digit = (uint32_t)b;
        s_rem = rem_g - fx_all;
        s_local_above = above_own + fx_own;
        s_tot_d = f_all;
      }
    }
    __syncthreads();
    local_greater += s_local_above;
    prefix = (prefix << bits) | s_digit;
    rem = s_rem;
    if (pass == 0 && p.cand && (uint32_t)k - rem + s_tot_d <= (uint32_t)kCand) {
      candidate_path(p, hist, cand, cached, half, cache16, keys4, len, c0, prefix, rem, local_greater, crank, csize,
                     out, w_gt, w_eq, w_selb, w_eqb, &s_cand_n, s_seg, &s_cbase, &s_digit, &s_rem);
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
  const int probe_smem = (3 * kBins + kMaxCacheKeys + 2 * kCand) * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, probe_smem);
  if (e != cudaSuccess) return e;
  int max_cluster = max_cluster_for(reinterpret_cast<const void*>(topk_kernel), kThreads, probe_smem,
                                    kClusterSlotTopk);
  if (max_cluster == 0) return cudaErrorUnknown;
  if (topk_cluster_cap() > 0) max_cluster = std::min(max_cluster, topk_cluster_cap());
  // cluster size: enough blocks per row that the rows fill a good share of the
  // GPU (each block reads less of the row), and chunks that fit the key cache
  // fewest blocks per row whose chunks fit the key cache -- whole keys, or,
  // when the rows outnumber what the GPU holds at once, the 16-bit key tops of
  // chunks twice as long (more rows in flight beats faster rows then)
  const bool many_rows = (int64_t)a.T * 2 > a.num_sms;
  const int fit = many_rows ? 2 * kMaxCacheKeys : kMaxCacheKeys;
  int c = 1;
  while (c < max_cluster && (a.max_n + c - 1) / c > fit) c *= 2;
  while (c < max_cluster && (int64_t)a.T * c * 2 <= a.num_sms && (a.max_n + 2 * c - 1) / (2 * c) >= 4096) c *= 2;
  const int per = (((a.max_n + c - 1) / c) + 7) & ~7;
  // the cache holds whole keys, or the top 16 bits of each key of a chunk up to twice as long
  const int cache_half = per > kMaxCacheKeys && per <= 2 * kMaxCacheKeys;
  const int cache_keys = per <= 2 * kMaxCacheKeys ? per : 0;
  const size_t cache_words = cache_half ? (size_t)cache_keys / 2 : (size_t)cache_keys;
  const size_t smem = (3 * kBins + cache_words + 2 * kCand) * 4;
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
  p.cache_half = cache_half;
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

// sparse_mla.cu -- sparse MLA in MQA mode over the selected latent rows.
//
// For query t and head h, over the selected positions s:
//   z_s = scale * Q[t, h, :D] . C[s, :D],  p = softmax(z),
//   O[t, h, :] = sum_s p_s C[s, :D_v],  LSE[t, h] = log sum_s exp(z_s)
// ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works /
// Model, sparse-MLA bullet: sparse MLA in MQA mode over the top-k tokens, all
// heads sharing the one latent row of a token).
//
// Layout of the work on the tensor cores.  128 selected rows are gathered into
// shared memory as D/64 column blocks of [128 rows x 64 dims] (128-byte
// swizzle).  The same bytes serve two MMAs:
//   S^T[key, h] = C[key, :] . Q[h, :]^T     M = 128 keys, N = 64 heads, K = D
//                 (C block K-major, Q block K-major)
//   O^T[v, h]  += C[key, v]^T . P^T[key, h] M = 128 value dims per block, N = 64
//                 heads, K = 128 keys (C block read MN-major, P MN-major)
// so the 64-head MQA tile is a real dense contraction with every TMEM lane in
// use (O^T: 4 x 64 columns, S^T: 64 columns).  One thread owns one key of S^T
// for 32 heads: the per-head softmax max over the 128 keys is a 31-shuffle
// transpose reduction per warp plus a 4-quadrant exchange; the running max is
// only raised when a head's max grows by more than 2^8 (the exact result is
// unchanged, only the reference point moves), so O^T is rarely rescaled.
//
// Row gather: for the 576-dim latent, TMA tile::gather4 moves four selected
// rows x 64 dims per instruction straight into the swizzled block, all nine
// blocks of a tile in flight at once, completion counted in bytes on one
// mbarrier per block.  (The 80-dim test latent uses 16-byte cp.async copies.)
//
// Split over a cluster: the selected rows of one query are divided among the
// blocks of a thread-block cluster; each block keeps its partial (m, l, O).
// The cluster combines them through distributed shared memory: each block
// pushes (remote stores, no round trips) its (m, l) to every block and its
// scaled partial output to the block owning each value slice, so partial
// outputs never travel through global memory.
//
// Warp roles (416 threads, one block per SM):
//   warps 0..3   row gather (index -> pool row, paged or contiguous)
//   warp 4       TMEM owner, query TMA, MMA issuer (one thread)
//   warps 5..12  softmax: two warps per TMEM lane quadrant, 32 heads each;
//                then the combine
#include <algorithm>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // raise the running max only past 2^8
constexpr int kSoftmaxThreads = 256;
constexpr int kMaxSplit = 8;  // blocks per cluster (splits of one query's rows)

template <int NB, int MB, bool PSEP, bool TMA4>
struct MlaCfg {
  static constexpr int THREADS = 160 + kSoftmaxThreads;
  static constexpr int BLK = 128 * 128;               // one [128 rows x 64 dims] block
  static constexpr int OFF_Q = 0;                     // NB x [64 heads x 64 dims]
  static constexpr int OFF_KV = OFF_Q + NB * 64 * 128;
  static constexpr int OFF_P = PSEP ? OFF_KV + NB * BLK : OFF_KV + (NB - 1) * BLK;
  static constexpr int OFF_ROWS = (PSEP ? OFF_P + BLK : OFF_KV + NB * BLK);  // 2 x 128 row pointers (cp.async)
  static constexpr int ROWS_BYTES = TMA4 ? 0 : 2 * 128 * 8;
  static constexpr int OFF_VALID = OFF_ROWS + ROWS_BYTES;                    // 2 x 128 int
  static constexpr int OFF_RED = OFF_VALID + 2 * 128 * 4;                    // 4 x 64 float
  static constexpr int OFF_MRUN = OFF_RED + 4 * 64 * 4;                      // 64 float
  static constexpr int OFF_ALPHA = OFF_MRUN + 64 * 4;                        // 64 float
  static constexpr int OFF_ML = OFF_ALPHA + 64 * 4;                          // 2 x 64 float (m, l)
  static constexpr int OFF_F = OFF_ML + 2 * 64 * 4;                          // 64 float
  static constexpr int OFF_MLT = OFF_F + 64 * 4;                             // [kMaxSplit][2][64] pushed (m, l)
  static constexpr int OFF_BAR = OFF_MLT + kMaxSplit * 2 * 64 * 4;
  static constexpr int N_BARS = 2 * NB + 8;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TMEM_COLS = (MB * 64 + 64) <= 128 ? 128 : (MB * 64 + 64) <= 256 ? 256 : 512;
  static constexpr int S_COL = MB * 64;
  static_assert(PSEP || NB > 2 * MB, "P reuses the last column block only when no value block lives there");
};

struct MlaParams {
  MlaLayerView layer[DSA_MAX_LAYERS];
  int32_t d_qk;
  int32_t d_v;
  const int32_t* idx;
  int64_t ld_idx;
  int32_t k;
  int32_t T;
  const int32_t* q_seq;
  const int32_t* q_n;
  int* err;
};

__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Per-lane reduction of 32 values across the warp by halving exchanges: lane l
// ends with the reduction over all 32 lanes of element l.
template <bool MAX>
__device__ __forceinline__ float transpose_reduce32(const float (&x)[32], int lane) {
  float y[16];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float keep = hi ? x[16 + i] : x[i];
      const float send = hi ? x[i] : x[16 + i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      y[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int w = 8, n = 8; w >= 1; w >>= 1, n >>= 1) {
    const bool hi = lane & w;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float keep = hi ? y[n + i] : y[i];
      const float send = hi ? y[i] : y[n + i];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      y[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return y[0];
}

template <int NB, int MB, bool PSEP, bool TMA4>
__global__ void __launch_bounds__(160 + kSoftmaxThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
                      const __grid_constant__ CUtensorMap tm_q2, const __grid_constant__ CUtensorMap tm_q3,
                      const __grid_constant__ CUtensorMap tm_c0, const __grid_constant__ CUtensorMap tm_c1,
                      const __grid_constant__ CUtensorMap tm_c2, const __grid_constant__ CUtensorMap tm_c3,
                      MlaParams p) {
  using C = MlaCfg<NB, MB, PSEP, TMA4>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const __nv_bfloat16** rows_s = reinterpret_cast<const __nv_bfloat16**>(smem + C::OFF_ROWS);
  int* valid_s = reinterpret_cast<int*>(smem + C::OFF_VALID);
  float* red_s = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* mrun_s = reinterpret_cast<float*>(smem + C::OFF_MRUN);
  float* alpha_s = reinterpret_cast<float*>(smem + C::OFF_ALPHA);
  float* ml_s = reinterpret_cast<float*>(smem + C::OFF_ML);
  float* f_s = reinterpret_cast<float*>(smem + C::OFF_F);
  float* mlt_s = reinterpret_cast<float*>(smem + C::OFF_MLT);  // [split][m or l][head]
  // combine buffers after the last tile (bf16 receive and staging areas)
  __nv_bfloat16* obuf_h = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_KV);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  auto bar_full = [&](int kb) { return smem_u32(bars + kb); };
  auto bar_empty = [&](int kb) { return smem_u32(bars + NB + kb); };
  const uint32_t bar_s_full = smem_u32(bars + 2 * NB);
  const uint32_t bar_p_full = smem_u32(bars + 2 * NB + 1);
  const uint32_t bar_q_full = smem_u32(bars + 2 * NB + 2);
  const uint32_t bar_o_done = smem_u32(bars + 2 * NB + 3);
  const uint32_t bar_drain = smem_u32(bars + 2 * NB + 4);
  auto bar_valid = [&](int par) { return smem_u32(bars + 2 * NB + 5 + par); };
  const uint32_t bar_recv = smem_u32(bars + 2 * NB + 7);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const int t = blockIdx.y % p.T;
  const int li = blockIdx.y / p.T;
  const MlaLayerView& L = p.layer[li];
  const CUtensorMap* tm_q = li == 0 ? &tm_q0 : li == 1 ? &tm_q1 : li == 2 ? &tm_q2 : &tm_q3;
  const CUtensorMap* tm_c = li == 0 ? &tm_c0 : li == 1 ? &tm_c1 : li == 2 ? &tm_c2 : &tm_c3;

  if (threadIdx.x == 0) {
    for (int kb = 0; kb < NB; ++kb) {
      mbar_init(bar_full(kb), TMA4 ? 1 : 128);
      mbar_init(bar_empty(kb), 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_p_full, kSoftmaxThreads);
    mbar_init(bar_q_full, 1);
    mbar_init(bar_o_done, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_valid(0), 128);
    mbar_init(bar_valid(1), 128);
    mbar_init(bar_recv, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (TMA4) prefetch_tmap(tm_c);
  }
  if (threadIdx.x >= 160 && threadIdx.x < 224) mrun_s[threadIdx.x - 160] = -INFINITY;
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the query is a caller input: its load may overlap the previous grid
  if (warp == 4 && lane == 0) {
    mbar_arrive_expect_tx(bar_q_full, NB * 64 * 128);
    for (int kb = 0; kb < NB; ++kb) tma_load_3d(sbase + C::OFF_Q + kb * 64 * 128, tm_q, bar_q_full, kb * 64, 0, t);
  }
  pdl_wait();  // positions and plan of the previous grids are complete from here on
  pdl_trigger();

  const int n_t = p.q_n[t];
  const int b = p.q_seq[t];
  const int nvalid = min(n_t, p.k);
  const int tiles = (nvalid + 127) / 128;
  const int j0 = (int)((int64_t)tiles * crank / csize), j1 = (int)((int64_t)tiles * (crank + 1) / csize);
  const int my_tiles = j1 - j0;

  if (warp < 4) {
    // ---------------------------------------------------------- row gather
    const int pt = threadIdx.x;              // key of the tile this thread resolves
    const int32_t* idx_row = p.idx + (int64_t)t * p.ld_idx;
    bool bad = false;
    for (int jj = 0; jj < my_tiles; ++jj) {
      const int j = j0 + jj;
      const int par = jj & 1;
      const uint32_t phase = jj & 1;
      int64_t row = -1;
      {
        const int e = j * 128 + pt;
        int pos = e < nvalid ? __ldg(idx_row + e) : -1;
        if (pos >= n_t || pos < -1) {
          atomicOr(p.err, DEV_ERR_BAD_INDEX);
          pos = -1;
        }
        if (pos >= 0) {
          row = cache_row(L.kv, b, pos);
          if (row < 0) atomicOr(p.err, DEV_ERR_BAD_INDEX);
        }
        valid_s[par * 128 + pt] = row >= 0;
        if (!TMA4) rows_s[par * 128 + pt] = row >= 0 ? L.kv.base + row * L.kv.row_stride : nullptr;
      }
      mbar_arrive(bar_valid(par));
      if constexpr (TMA4) {
        // lanes 0..7 of warp w gather rows 32w + 4l .. +3; an unused slot reads
        // pool row 0 (finite data; its probability is zero)
        const int32_t rr = row >= 0 ? (int32_t)row : 0;
        const int src = (lane & 7) * 4;
        const int32_t r0 = __shfl_sync(0xffffffffu, rr, src), r1 = __shfl_sync(0xffffffffu, rr, src + 1);
        const int32_t r2 = __shfl_sync(0xffffffffu, rr, src + 2), r3 = __shfl_sync(0xffffffffu, rr, src + 3);
        if (lane < 8) {
          const uint32_t dst_off = (uint32_t)(warp * 8 + lane) * 512;
#pragma unroll 1
          for (int kb = 0; kb < NB; ++kb) {
            bad |= !mbar_wait(bar_empty(kb), phase ^ 1, abort_flag, p.err);
            if (warp == 0 && lane == 0) mbar_arrive_expect_tx(bar_full(kb), C::BLK);
            if (!bad)
              tma_gather4(sbase + C::OFF_KV + kb * C::BLK + dst_off, tm_c, bar_full(kb), kb * 64, r0, r1, r2, r3);
          }
        }
        // lanes 8..31 wait here for the issuing lanes: nobody may rewrite this
        // tile parity's valid flags before the empties of the next tile came back
        __syncwarp();
      } else {
        named_bar_sync(2, 128);
        const int chunk = pt & 7;
#pragma unroll 1
        for (int kb = 0; kb < NB; ++kb) {
          bad |= !mbar_wait(bar_empty(kb), phase ^ 1, abort_flag, p.err);
          if (!bad) {
            const uint32_t dst0 = sbase + C::OFF_KV + kb * C::BLK;
            const int col = kb * 64 + chunk * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = (pt >> 3) + 16 * i;
              const __nv_bfloat16* src = rows_s[par * 128 + r];
              const bool ok = src != nullptr && col < p.d_qk;
              cp_async_16(dst0 + r * 128 + ((chunk ^ (r & 7)) << 4),
                          ok ? (const void*)(src + col) : (const void*)L.kv.base, ok ? 16u : 0u);
            }
          }
          cp_async_commit();
          if (kb >= 2) {  // signal the block issued two steps ago once its copies have landed
            cp_async_wait_group<2>();
            fence_proxy_async_smem();
            mbar_arrive(bar_full(kb - 2));
          }
        }
        cp_async_wait_group<0>();
        fence_proxy_async_smem();
        for (int kb = (NB >= 2 ? NB - 2 : 0); kb < NB; ++kb) mbar_arrive(bar_full(kb));
      }
    }
    if (!TMA4) cp_async_wait_all();
  } else if (warp == 4) {
    // ---------------------------------------------- query TMA + MMA issuer
    if (lane == 0) {
      bool bad = !mbar_wait(bar_q_full, 0, abort_flag, p.err);
      if (bad) mbar_wait_drain(bar_q_full, 0);  // the query copy lands before the block may exit
      constexpr uint32_t idesc_s = mma_idesc_bf16(128, 64, false, false);
      constexpr uint32_t idesc_o = mma_idesc_bf16(128, 64, true, true);
      for (int jj = 0; jj < my_tiles && !bad; ++jj) {
        const uint32_t phase = jj & 1;
        // S^T = C . Q^T over all D/64 column blocks
        for (int kb = 0; kb < NB && !bad; ++kb) {
          if (!mbar_wait(bar_full(kb), phase, abort_flag, p.err)) { bad = true; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc_sw128(sbase + C::OFF_KV + kb * C::BLK + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(sbase + C::OFF_Q + kb * 64 * 128 + kk * 32, 16, 1024);
            mma_bf16(tmem + C::S_COL, ad, bd, idesc_s, (kb | kk) != 0);
          }
        }
        if (bad) break;
        mma_commit(bar_s_full);
        for (int kb = 2 * MB; kb < NB; ++kb)
          if (PSEP || kb != NB - 1) mma_commit(bar_empty(kb));  // blocks read by S only
        // O^T += C^T . P^T over the 128 keys
        if (!mbar_wait(bar_p_full, phase, abort_flag, p.err)) { bad = true; break; }
        tc_fence_after();
        for (int mb = 0; mb < MB; ++mb) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = smem_desc_sw128(sbase + C::OFF_KV + 2 * mb * C::BLK + kk * 2048, C::BLK, 1024);
            const uint64_t bd = smem_desc_sw128(sbase + C::OFF_P + kk * 2048, C::BLK, 1024);
            mma_bf16(tmem + mb * 64, ad, bd, idesc_o, (jj | kk) != 0);
          }
          mma_commit(bar_empty(2 * mb));
          if (2 * mb + 1 < NB) mma_commit(bar_empty(2 * mb + 1));
        }
        if (!PSEP) mma_commit(bar_empty(NB - 1));
      }
      mma_commit(bar_o_done);
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int quad = warp & 3;
    const int half = (warp - 5) >> 2;        // heads 32*half .. +31
    const int row = quad * 32 + lane;        // key (S^T) or value dim (O^T) lane
    const int st = threadIdx.x - 160;        // 0..255
    const int h0 = half * 32;
    const float c = L.scale * kLog2e;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    float lsum[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) lsum[i] = 0.f;
    bool bad = false;
    for (int jj = 0; jj < my_tiles; ++jj) {
      const int par = jj & 1;
      bad |= !mbar_wait(bar_valid(par), (jj >> 1) & 1, abort_flag, p.err);
      const bool kv = valid_s[par * 128 + row] != 0;
      bad |= !mbar_wait(bar_s_full, par, abort_flag, p.err);
      tc_fence_after();
      float x[32];
      {
        uint32_t r[32];
        tmem_ld32(lane_base + C::S_COL + h0, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = kv ? __uint_as_float(r[i]) * c : -INFINITY;
      }
      // per-head max over this warp's 32 keys; lane l ends with head h0 + l
      red_s[quad * 64 + h0 + lane] = transpose_reduce32<true>(x, lane);
      named_bar_sync(3, kSoftmaxThreads);
      bool rescale = false;
      if (st < 64) {
        const float mt = fmaxf(fmaxf(red_s[st], red_s[64 + st]), fmaxf(red_s[128 + st], red_s[192 + st]));
        const float mr = mrun_s[st];
        float alpha = 1.f;
        if (mt > mr + kRescaleLog2 || (mr == -INFINITY && mt > -INFINITY)) {
          alpha = (mr == -INFINITY) ? 0.f : exp2f(mr - mt);
          mrun_s[st] = mt;
          rescale = mr != -INFINITY;
        }
        alpha_s[st] = alpha;
      }
      rescale = bar_red_or(4, kSoftmaxThreads, rescale);
      // probabilities, running sums, this key's P^T row for heads h0..h0+31 (bf16).
      // Without a rescale every alpha is 1 (or the sum is still 0), so the
      // running sums only add.
      if (rescale) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(alpha_s + h0 + i);
          lsum[i] *= a4.x; lsum[i + 1] *= a4.y; lsum[i + 2] *= a4.z; lsum[i + 3] *= a4.w;
        }
      }
      const uint32_t prow = sbase + C::OFF_P + row * 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float pv[8], mref[8];
        {
          const float4 ma = *reinterpret_cast<const float4*>(mrun_s + h0 + cc * 8);
          const float4 mb4 = *reinterpret_cast<const float4*>(mrun_s + h0 + cc * 8 + 4);
          mref[0] = ma.x; mref[1] = ma.y; mref[2] = ma.z; mref[3] = ma.w;
          mref[4] = mb4.x; mref[5] = mb4.y; mref[6] = mb4.z; mref[7] = mb4.w;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = cc * 8 + j;
          pv[j] = x[i] == -INFINITY ? 0.f : exp2f(x[i] - mref[j]);  // no valid key yet: m is -inf too
          lsum[i] += pv[j];
        }
        const int chunk = half * 4 + cc;
        st_shared_v4(prow + ((chunk ^ (row & 7)) << 4), pack_bf16x2(pv[0], pv[1]), pack_bf16x2(pv[2], pv[3]),
                     pack_bf16x2(pv[4], pv[5]), pack_bf16x2(pv[6], pv[7]));
      }
      fence_proxy_async_smem();
      if (rescale && !bad) {
        // move O^T to the new reference point: column h times alpha[h]
        for (int mb = 0; mb < MB; ++mb) {
          uint32_t r[32];
          tmem_ld32(lane_base + mb * 64 + h0, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha_s[h0 + i]);
          tmem_st32(lane_base + mb * 64 + h0, r);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(bar_p_full);
      named_bar_sync(3, kSoftmaxThreads);  // alpha_s / mrun_s / red_s are rewritten by the next tile
    }
    // l per head over this block's keys
    red_s[quad * 64 + h0 + lane] = transpose_reduce32<false>(lsum, lane);
    named_bar_sync(3, kSoftmaxThreads);
    if (st < 64) {
      ml_s[st] = mrun_s[st];
      ml_s[64 + st] = red_s[st] + red_s[64 + st] + red_s[128 + st] + red_s[192 + st];
    }
    if (my_tiles > 0) bad |= !mbar_wait(bar_o_done, 0, abort_flag, p.err);
    tc_fence_after();
  }

  // ------------------------------------------------- combine over the cluster
  // Push model: every block stores its (m, l) per head into every block's
  // table, then its scaled partial output straight into the shared memory of
  // the block that owns each value slice; remote stores do not wait for a
  // round trip, and no block reads another block's memory.
  __syncthreads();
  if (threadIdx.x >= 160 && threadIdx.x < 224) {
    const int h = threadIdx.x - 160;
    const float m_own = ml_s[h], l_own = ml_s[64 + h];
    for (uint32_t r = 0; r < csize; ++r) {
      st_dsmem_f32(dsmem_addr(smem_u32(mlt_s + (crank * 2 + 0) * 64 + h), r), m_own);
      st_dsmem_f32(dsmem_addr(smem_u32(mlt_s + (crank * 2 + 1) * 64 + h), r), l_own);
    }
  }
  cluster_sync();  // every table complete; every block is past its main loop
  if (threadIdx.x >= 160 && threadIdx.x < 224) {
    const int h = threadIdx.x - 160;
    float M = -INFINITY;
    for (uint32_t r = 0; r < csize; ++r) M = fmaxf(M, mlt_s[(r * 2) * 64 + h]);
    float Lsum = 0.f;
    if (M != -INFINITY)
      for (uint32_t r = 0; r < csize; ++r) {
        const float m_r = mlt_s[(r * 2) * 64 + h];
        if (m_r != -INFINITY) Lsum += mlt_s[(r * 2 + 1) * 64 + h] * exp2f(m_r - M);
      }
    const float m_own = ml_s[h];
    f_s[h] = (Lsum > 0.f && m_own != -INFINITY) ? exp2f(m_own - M) / Lsum : 0.f;
    if (crank == 0 && L.lse != nullptr && h < L.H)
      L.lse[(int64_t)t * L.H + h] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  // Scaled partial outputs in bf16, [source block][head][value dim of the
  // owner's slice]: this block's own slice goes straight into its receive
  // area, the others into a staging area, one contiguous slice per owner, and
  // the TMA engine copies each staged slice into its owner's receive area.
  const int slice = p.d_v / (int)csize;
  const int rs = slice + 8;  // head row stride (16 bytes of padding spread the banks)
  const uint32_t slice_bytes = 64u * (uint32_t)rs * 2u;
  __nv_bfloat16* recv_h = obuf_h;                                 // [csize][64][rs]
  __nv_bfloat16* send_h = obuf_h + (size_t)csize * 64 * rs;       // [csize][64][rs]
  if (warp >= 5) {
    const int quad = warp & 3;
    const int h0 = ((warp - 5) >> 2) * 32;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    // The query tile is dead now: each warp transposes 16 heads x 32 value
    // dims there so that one thread writes 8 consecutive value dims of a head.
    float* stage = reinterpret_cast<float*>(smem + C::OFF_Q) + (warp - 5) * 512;
    for (int mb = 0; mb < MB; ++mb) {
      uint32_t r[32];
      if (my_tiles > 0) {
        tmem_ld32(lane_base + mb * 64 + h0, r);
        tmem_wait_ld();
      }
      const int vq = mb * 128 + quad * 32;  // this warp's first value dim (warp-uniform)
      if (vq < p.d_v) {
        const int owner = vq / slice;
        const int vvq = vq - owner * slice;
        __nv_bfloat16* dst = owner == (int)crank ? recv_h + (size_t)crank * 64 * rs
                                                 : send_h + (size_t)owner * 64 * rs;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int h = h0 + hh * 16 + j;
            stage[j * 32 + lane] = my_tiles > 0 ? __uint_as_float(r[hh * 16 + j]) * f_s[h] : 0.f;
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // a warp reads 4 heads' 32 value dims (512 contiguous bytes)
            const int hl = k * 4 + (lane >> 3), c4 = lane & 7;
            const float4 a4 = *reinterpret_cast<const float4*>(stage + hl * 32 + 4 * c4);
            const int h = h0 + hh * 16 + hl;
            st_shared_v2(smem_u32(dst + h * rs + vvq + 4 * c4), pack_bf16x2(a4.x, a4.y), pack_bf16x2(a4.z, a4.w));
          }
          __syncwarp();
        }
      }
    }
    fence_proxy_async_smem();  // staged slices are read by the TMA engine next
  }
  __syncthreads();
  if (threadIdx.x == 160 && csize > 1) {
    mbar_arrive_expect_tx(bar_recv, (csize - 1) * slice_bytes);
    for (uint32_t o = 0; o < csize; ++o) {
      if (o == crank) continue;
      bulk_copy_smem_to_peer(dsmem_addr(smem_u32(recv_h + (size_t)crank * 64 * rs), o),
                             smem_u32(send_h + (size_t)o * 64 * rs), slice_bytes, dsmem_addr(bar_recv, o));
    }
  }
  if (csize > 1) {
    bool ok = true;
    if (warp >= 5) ok = mbar_wait(bar_recv, 0, abort_flag, p.err);  // every peer's slice has landed
    (void)ok;
    __syncthreads();
  }
  {
    const int v0 = (int)crank * slice;
    const int per_h = slice / 4;
    const int items = L.H * per_h;
    for (int it = threadIdx.x; it < items; it += C::THREADS) {
      const int h = it / per_h;
      const int vv = (it % per_h) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t r = 0; r < csize; ++r) {
        const uint2 o = *reinterpret_cast<const uint2*>(recv_h + ((int)r * 64 + h) * rs + vv);
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.y));
        acc.x += lo.x; acc.y += lo.y; acc.z += hi.x; acc.w += hi.y;
      }
      uint2 packed;
      packed.x = pack_bf16x2(acc.x, acc.y);
      packed.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(L.out + ((int64_t)t * L.H + h) * p.d_v + v0 + vv) = packed;
    }
  }
  // no block may leave while a peer's copy could still read its staging area
  if (csize > 1) cluster_sync();
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

int g_max_cluster_mla[2] = {0, 0};

template <int NB, int MB, bool PSEP, bool TMA4>
cudaError_t launch_t(const MlaLaunch& a, cudaStream_t stream, int which) {
  using C = MlaCfg<NB, MB, PSEP, TMA4>;
  auto kern = sparse_mla_kernel<NB, MB, PSEP, TMA4>;
  CUtensorMap tq[DSA_MAX_LAYERS], tc[DSA_MAX_LAYERS];
  for (int l = 0; l < DSA_MAX_LAYERS; ++l) {
    const int ls = l < a.n_layers ? l : 0;
    const MlaLayerView& lv = a.layer[ls];
    {
      const uint64_t dims[3] = {(uint64_t)a.d_qk, (uint64_t)lv.H, (uint64_t)a.T};
      const uint64_t strides[2] = {(uint64_t)a.d_qk * 2, (uint64_t)a.d_qk * lv.H * 2};
      const uint32_t box[3] = {64u, 64u, 1u};
      if (encode_tmap(&tq[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, lv.q, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    if (TMA4) {
      const uint64_t dims[2] = {(uint64_t)a.d_qk, (uint64_t)lv.kv.num_rows};
      const uint64_t strides[1] = {(uint64_t)lv.kv.row_stride * 2};
      const uint32_t box[2] = {64u, 1u};
      if (encode_tmap(&tc[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lv.kv.base, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    } else {
      tc[l] = tq[l];  // unused by the cp.async gather
    }
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (g_max_cluster_mla[which] == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    g_max_cluster_mla[which] = 8;
    cudaLaunchConfig_t probe = {};
    probe.gridDim = dim3(16, 1, 1);
    probe.blockDim = dim3(C::THREADS, 1, 1);
    probe.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 16;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    probe.attrs = &at;
    probe.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &probe) == cudaSuccess && nclusters > 0)
      g_max_cluster_mla[which] = 16;
    cudaGetLastError();
  }
  const int units = a.T * a.n_layers;
  const int tiles_max = (std::min(a.k, a.max_n) + 127) / 128;
  int c = 1;
  while (c * 2 <= std::min(g_max_cluster_mla[which], kMaxSplit) && c * 2 <= tiles_max && (int64_t)units * c * 2 <= a.num_sms)
    c *= 2;
  // every block owns a value slice of >= 32 dims (one warp's rows push to one owner)
  while (c > 1 && (a.d_v % (32 * c) != 0)) c /= 2;

  MlaParams p;
  for (int l = 0; l < DSA_MAX_LAYERS; ++l) p.layer[l] = a.layer[l < a.n_layers ? l : 0];
  p.d_qk = a.d_qk;
  p.d_v = a.d_v;
  p.idx = a.idx;
  p.ld_idx = a.ld_idx;
  p.k = a.k;
  p.T = a.T;
  p.q_seq = a.q_seq;
  p.q_n = a.q_n;
  p.err = a.err;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c, units, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = c;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1] = pdl_attribute();
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tq[0], tq[1], tq[2], tq[3], tc[0], tc[1], tc[2], tc[3], p);
}

}  // namespace

cudaError_t launch_sparse_mla(const MlaLaunch& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  if (a.d_qk == 576 && a.d_v == 512) return launch_t<9, 4, false, true>(a, stream, 0);
  if (a.d_qk == 80 && a.d_v == 64) return launch_t<2, 1, true, false>(a, stream, 1);
  return cudaErrorInvalidValue;
}

}  // namespace dsa

// sparse_mha.cu -- MHA mode of sparse attention: per-head keys and values
// up-projected from the latent rows, softmax attention of every head over the
// top-k selection of its query.
//
// "How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works /
// Model, second bullet: sparse MLA runs in MQA mode, and vLLM switches to MHA
// mode for contexts of about 2K-5K tokens.  MQA mode reads one 576-dim latent
// row per selected token with the up-projections absorbed into the query and
// the output; MHA mode up-projects every token of a short context once and
// attends with per-head keys (192 no-rope dims + the 64 shared rope dims) and
// values (256 dims), which pays off when many queries -- a prefill chunk --
// share that context.
//
// Three kernels:
//   project  K[r, h] = (W_UK[h] c[r, :512], c[r, 512:576]) and
//            V[r, h] = W_UV[h] c[r, :512] for every row r of a latent pool: a
//            tcgen05 GEMM per (128 rows, head), A = the latent rows (TMA,
//            128-byte swizzle), B = the head's projection rows, fp32 in TMEM,
//            bf16 rows written by the epilogue (keys also copy the rope dims)
//   mask     the selection of every query as a bit mask over its positions
//            (one block per query, built in shared memory)
//   attend   one block per (group of up to 128 consecutive queries of one
//            sequence, head), keys in tiles of 64 positions (one 64-token
//            page): S = Q K^T (M = 128 queries, N = 64 keys, K = 256) into one
//            of two TMEM buffers, online softmax in fp32 over the selected
//            keys only (a per-row reference that moves when a score passes it
//            by more than 2^8, so O is rescaled in TMEM only then), P in bf16
//            into one of two tensor-memory buffers (each thread its own lane),
//            O += P V (M = 128, N = 256, K = 64) with P read from tensor memory.  Warp 0 streams Q once and K/V tiles through two stages
//            with TMA, warp 1 issues the MMAs, warps 2-9 do the softmax: two
//            threads per query row, both finding the row maximum over the
//            tile's 64 keys, each exponentiating 32 of them and owning 128 of
//            the row's output columns.
#include <algorithm>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kLatent = 512;  // latent dims the projections read (the rest are rope dims)
constexpr int kRope = 64;
constexpr int kHead = 256;    // per-head q/k dims (no-rope + rope) and value dims of the kernels

// ------------------------------------------------------------ project ---

template <int N>
struct ProjCfg {
  static constexpr int STAGES = 4;
  static constexpr int KB = kLatent / 64;        // 64-dim K blocks
  static constexpr int A_BYTES = 128 * 128;      // 128 rows x 64 dims
  static constexpr int B_BYTES = N * 128;        // N outputs x 64 dims
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int THREADS = 64 + 128;       // producer, MMA issuer, four epilogue warps
  static constexpr int N_BARS = 2 * STAGES + 4 + 1;
  static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static_assert(N % 16 == 0 && N <= 256, "tcgen05 M=128 needs N in [16, 256]");
  static_assert(SMEM_BYTES <= 227 * 1024, "projection stages exceed shared memory");
};

struct ProjParams {
  const __nv_bfloat16* c;  // latent pool [rows, c_stride]
  int64_t c_stride;
  int64_t rows;
  int32_t H;
  __nv_bfloat16* out;      // [rows, H, kHead]
  int* err;
};

// Persistent: one block per SM walks the (128-row tile, head) output tiles
// t = blockIdx.x, + gridDim.x, ...  The producer streams the tiles' K blocks
// (latent rows and the head's projection rows) through a ring of stages
// across tile boundaries; the MMA issuer accumulates each tile into one of two
// TMEM accumulators, so the epilogue of one tile (four warps, one row a
// thread) overlaps the MMAs of the next.
template <int N, bool KEYS>
__global__ void __launch_bounds__(ProjCfg<N>::THREADS, 1)
    mha_project_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_w,
                       ProjParams p) {
  using C = ProjCfg<N>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + C::STAGES + s); };
  auto acc_full = [&](int a) { return smem_u32(bars + 2 * C::STAGES + a); };
  auto acc_empty = [&](int a) { return smem_u32(bars + 2 * C::STAGES + 2 + a); };
  const uint32_t drain = smem_u32(bars + 2 * C::STAGES + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_rt = (int)((p.rows + 127) / 128);
  const int n_tiles = n_rt * p.H;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_c);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * N <= 256 ? 256 : 512);
    tmem_relinquish();
  }
  pdl_wait();  // the latent pool may come from the previous kernel on the stream
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;  // K blocks issued, over all of this block's tiles
      for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
        const int r0 = (t / p.H) * 128, h = t % p.H;
        for (int kb = 0; kb < C::KB; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (it >= C::STAGES && !mbar_wait(empty(s), ((it / C::STAGES) - 1) & 1, abort_flag, p.err)) break;
          const uint32_t dst = sbase + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(full(s), C::STAGE_BYTES);
          tma_load_2d(dst, &tm_c, full(s), kb * 64, r0);
          tma_load_2d(dst + C::A_BYTES, &tm_w, full(s), kb * 64, h * N);
        }
      }
      if (*abort_flag)  // the loads already issued land before the block leaves
        for (int j = std::max(0, it - C::STAGES); j < it; ++j)
          mbar_wait_drain(full(j % C::STAGES), (j / C::STAGES) & 1);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = mma_idesc_bf16(128, N, false, false);
      bool ok = true;
      int it = 0, i = 0;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++i) {
        const int a = i & 1;
        // the epilogue has read this accumulator's previous tile
        if (i >= 2 && !(ok = mbar_wait(acc_empty(a), ((i >> 1) - 1) & 1, abort_flag, p.err))) break;
        tc_fence_after();
        for (int kb = 0; kb < C::KB; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (!(ok = mbar_wait(full(s), (it / C::STAGES) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          const uint32_t a0 = sbase + s * C::STAGE_BYTES, b0 = a0 + C::A_BYTES;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + a * N, smem_desc_sw128(a0 + ks * 32, 16, 1024), smem_desc_sw128(b0 + ks * 32, 16, 1024),
                     idesc, (kb | ks) != 0);
          mma_commit(empty(s));
        }
        if (ok) mma_commit(acc_full(a));
      }
      mma_commit(drain);  // every MMA of this thread done before TMEM is freed
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------------------------------------------- epilogue: one row a thread
    const int quad = warp & 3;  // TMEM lanes 32 * quad .. + 31
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
      const int a = i & 1;
      if (!mbar_wait(acc_full(a), (i >> 1) & 1, abort_flag, p.err)) break;
      tc_fence_after();
      const int h = t % p.H;
      const int64_t r = (int64_t)(t / p.H) * 128 + row;
#pragma unroll 1
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(lane_base + a * N + c0, v);
        tmem_wait_ld();
        if (r < p.rows) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + (r * p.H + h) * kHead + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty(a));  // the accumulator may take the tile after next
      if (KEYS && r < p.rows) {   // the rope dims every head shares follow the head's no-rope dims
        const uint4* src = reinterpret_cast<const uint4*>(p.c + r * p.c_stride + kLatent);
        uint4* dst = reinterpret_cast<uint4*>(p.out + (r * p.H + h) * kHead + N);
#pragma unroll
        for (int q = 0; q < kRope / 8; ++q) dst[q] = __ldg(src + q);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * N <= 256 ? 256 : 512);
  }
}

// ---------------------------------------------------------------- mask ---

struct MaskParams {
  const int32_t* idx;
  int64_t ld_idx;
  int32_t k;
  int32_t T;
  int32_t W;  // words per query row
  const int32_t* q_n;
  uint32_t* mask;
  int* err;
};

__global__ void __launch_bounds__(256) mha_mask_kernel(MaskParams p) {
  extern __shared__ uint32_t bits[];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  for (int i = threadIdx.x; i < p.W; i += blockDim.x) bits[i] = 0;
  __syncthreads();
  const int n_t = p.q_n[t];
  const int m = min(n_t, p.k);
  for (int j = threadIdx.x; j < m; j += blockDim.x) {
    const int pos = p.idx[(int64_t)t * p.ld_idx + j];
    if (pos == -1) continue;
    if (pos < -1 || pos >= n_t) {
      atomicOr(p.err, DEV_ERR_BAD_INDEX);
      continue;
    }
    atomicOr(bits + (pos >> 5), 1u << (pos & 31));
  }
  __syncthreads();
  uint32_t* dst = p.mask + (int64_t)t * p.W;
  for (int i = threadIdx.x; i < p.W; i += blockDim.x) dst[i] = bits[i];
}

// -------------------------------------------------------------- attend ---

struct AttCfg {
  static constexpr int THREADS = 64 + 256;               // producer, MMA issuer, eight softmax warps
  static constexpr int Q_BYTES = 128 * kHead * 2;        // 64 KB: 4 blocks [128 x 64]
  static constexpr int K_BYTES = 64 * kHead * 2;         // 32 KB: 4 blocks [64 x 64]
  static constexpr int V_BYTES = 64 * kHead * 2;         // 32 KB: 4 value blocks [64 keys x 64]
  static constexpr int K_STAGES = 3;
  static constexpr int V_STAGES = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + K_STAGES * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + V_STAGES * V_BYTES;
  static constexpr int N_BARS = 20;
  static constexpr int OFF_MISC = OFF_BAR + 8 * N_BARS;
  static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t S_COL = 256;                 // O: columns 0..255; S: two buffers of 64
  static constexpr uint32_t P_COL = 384;                 // P: two buffers of 32 (64 keys, bf16 pairs)
};

struct AttParams {
  PlanView plan;
  CacheView kv;           // addressing of the per-head key / value caches (rows of H x 256)
  const uint32_t* mask;
  int32_t W;
  int32_t H;
  float scale_log2;
  __nv_bfloat16* out;     // [T, H, kHead]
  float* lse;             // [T, H] or null
  int* err;
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__global__ void __launch_bounds__(AttCfg::THREADS, 1)
    mha_attend_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, AttParams p) {
  using C = AttCfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const uint32_t q_full = smem_u32(bars + 0);
  auto k_full = [&](int s) { return smem_u32(bars + 1 + s); };    // 3
  auto k_empty = [&](int s) { return smem_u32(bars + 4 + s); };   // 3
  auto v_full = [&](int s) { return smem_u32(bars + 7 + s); };    // 2
  auto v_empty = [&](int s) { return smem_u32(bars + 9 + s); };   // 2
  auto s_full = [&](int u) { return smem_u32(bars + 11 + u); };
  auto s_free = [&](int u) { return smem_u32(bars + 13 + u); };
  auto p_full = [&](int u) { return smem_u32(bars + 15 + u); };
  auto pv_done = [&](int u) { return smem_u32(bars + 17 + u); };
  const uint32_t drain = smem_u32(bars + 19);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();  // the plan and the masks are complete from here on
  pdl_trigger();
  // groups in reverse: a sequence's later groups see more keys (causal), so the
  // longest blocks start first and the short ones fill the last wave
  const int g = p.plan.header[0] - 1 - (int)blockIdx.x, h = blockIdx.y;
  if (g < 0) return;  // the grid is sized for the most groups a batch can have
  const int4 gi = p.plan.g_info[g];   // {sequence, first query, queries, n of the last query}
  const int b = gi.x, q0 = gi.y, cnt = gi.z;
  const int n_kt = (gi.w + 63) / 64;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::K_STAGES; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_free(s), 256);
      mbar_init(p_full(s), 256);
      mbar_init(pv_done(s), 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  // value stages start as zeros: a key that no query selects contributes P = 0
  // times whatever its stage holds, which must not be a NaN pattern
  for (int i = threadIdx.x; i < C::V_STAGES * C::V_BYTES / 16; i += C::THREADS)
    st_shared_v4(sbase + C::OFF_V + i * 16, 0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kt > 0) {
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      for (int kb = 0; kb < 4; ++kb) tma_load_3d(sbase + C::OFF_Q + kb * 16384, &tm_q, q_full, kb * 64, h, q0);
      // keys and values have stages of their own: a key stage is free once
      // its S = Q K^T is done, a value stage only after its P.V, so keys (three
      // stages) are loaded two tiles ahead of values (two stages).  A 64-key
      // tile is one 64-token page.
      const int32_t* pt = p.kv.paged ? p.kv.page_table + (int64_t)b * p.kv.pt_stride : nullptr;
      const int64_t start = p.kv.paged ? 0 : __ldg(p.kv.seq_start + b);
      int64_t row_of[3] = {0, 0, 0};
      bool valid_of[3] = {false, false, false};
      int issued_k = 0, issued_v = 0;
      auto issue_k = [&](int j) -> bool {
        const int s = j % 3;
        int64_t row0;
        bool valid;
        if (p.kv.paged) {
          const int64_t phys = __ldg(pt + j);
          valid = phys >= 0 && (phys + 1) * 64 <= p.kv.num_rows;
          row0 = phys * 64;
        } else {
          row0 = start + (int64_t)j * 64;
          valid = row0 >= 0 && row0 < p.kv.num_rows;
        }
        row_of[s] = row0;
        valid_of[s] = valid;
        if (j >= 3 && !mbar_wait(k_empty(s), ((j / 3) - 1) & 1, abort_flag, p.err)) return false;
        const uint32_t dst = sbase + C::OFF_K + s * C::K_BYTES;
        if (valid) {
          mbar_arrive_expect_tx(k_full(s), C::K_BYTES);
          for (int kb = 0; kb < 4; ++kb) tma_load_3d(dst + kb * 8192, &tm_k, k_full(s), kb * 64, h, (int32_t)row0);
        } else {
          atomicOr(p.err, DEV_ERR_BAD_INDEX);
          mbar_arrive(k_full(s));  // nothing loaded: the stage keeps earlier (finite) contents
        }
        ++issued_k;
        return true;
      };
      auto issue_v = [&](int j) -> bool {
        const int s = j & 1, r = j % 3;
        if (j >= 2 && !mbar_wait(v_empty(s), ((j >> 1) - 1) & 1, abort_flag, p.err)) return false;
        const uint32_t dst = sbase + C::OFF_V + s * C::V_BYTES;
        if (valid_of[r]) {
          mbar_arrive_expect_tx(v_full(s), C::V_BYTES);
          for (int kb = 0; kb < 4; ++kb)
            tma_load_3d(dst + kb * 8192, &tm_v, v_full(s), kb * 64, h, (int32_t)row_of[r]);
        } else {
          mbar_arrive(v_full(s));
        }
        ++issued_v;
        return true;
      };
      if (issue_k(0) && (n_kt < 2 || issue_k(1))) {
        for (int j = 0; j < n_kt; ++j) {
          if (j + 2 < n_kt && !issue_k(j + 2)) break;
          if (!issue_v(j)) break;
        }
      }
      if (*abort_flag) {
        mbar_wait_drain(q_full, 0);
        for (int j = std::max(0, issued_k - 3); j < issued_k; ++j) mbar_wait_drain(k_full(j % 3), (j / 3) & 1);
        for (int j = std::max(0, issued_v - 2); j < issued_v; ++j) mbar_wait_drain(v_full(j & 1), (j >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0 && n_kt > 0) {
      const uint32_t idesc_s = mma_idesc_bf16(128, 64, false, false);
      const uint32_t idesc_o = mma_idesc_bf16(128, kHead, false, true);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.err);
      auto issue_s = [&](int j) {
        const int u = j & 1, ks3 = j % 3;
        const uint32_t kbase = sbase + C::OFF_K + ks3 * C::K_BYTES;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + C::S_COL + u * 64, smem_desc_sw128(sbase + C::OFF_Q + kb * 16384 + ks * 32, 16, 1024),
                     smem_desc_sw128(kbase + kb * 8192 + ks * 32, 16, 1024), idesc_s, (kb | ks) != 0);
        mma_commit(k_empty(ks3));
        mma_commit(s_full(u));
      };
      auto issue_pv = [&](int j) {
        const int u = j & 1;
        const uint32_t vbase = sbase + C::OFF_V + u * C::V_BYTES;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // P from tensor memory: 16 keys = 8 columns per step
          mma_bf16_ts(tmem, tmem + C::P_COL + u * 32 + ks * 8, smem_desc_sw128(vbase + ks * 2048, 8192, 1024),
                      idesc_o, (j | ks) != 0);
        mma_commit(v_empty(u));
        mma_commit(pv_done(u));
      };
      auto ready_s = [&](int j) {
        const int u = j & 1;
        return mbar_test_wait(k_full(j % 3), (j / 3) & 1) &&
               (j < 2 || mbar_test_wait(s_free(u), ((j >> 1) - 1) & 1));
      };
      auto ready_pv = [&](int j) {
        const int u = j & 1;
        return mbar_test_wait(p_full(u), (j >> 1) & 1) && mbar_test_wait(v_full(u), (j >> 1) & 1);
      };
      if (ok && (ok = mbar_wait(k_full(0), 0, abort_flag, p.err))) {
        tc_fence_after();
        issue_s(0);
      }
      // per tile: the next tile's S and this tile's P.V, whichever is ready first
      for (int j = 0; j < n_kt && ok; ++j) {
        bool need_s = j + 1 < n_kt, need_pv = true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t spin = 1; need_s || need_pv; ++spin) {
          if (need_s && ready_s(j + 1)) {
            tc_fence_after();
            issue_s(j + 1);
            need_s = false;
          } else if (need_pv && ready_pv(j)) {
            tc_fence_after();
            issue_pv(j);
            need_pv = false;
          } else if ((spin & 31) == 0) {
            if (*abort_flag) {
              ok = false;
              break;
            }
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
              *abort_flag = 1;
              atomicOr(p.err, DEV_ERR_TIMEOUT);
              ok = false;
              break;
            }
          }
        }
      }
      mma_commit(drain);  // every MMA of this thread done before TMEM is freed
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------------------------------- softmax, two threads per query row
    const int qd = warp & 3;
    const int hf = (warp - 2) >> 2;  // which half of the tile's keys / of the row's outputs
    const int row = qd * 32 + lane;
    const int t = q0 + row;
    const bool valid_q = row < cnt;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t* mrow = p.mask + (int64_t)(valid_q ? t : 0) * p.W;
    float m_ref = neg_inf(), l = 0.f;  // l: this thread's half of the row sum
    bool ok = true;
    // the selection bits of a tile are loaded one tile ahead, so their latency
    // hides behind the previous tile
    uint2 bits_next = (valid_q && n_kt > 0) ? __ldg(reinterpret_cast<const uint2*>(mrow)) : make_uint2(0u, 0u);
    for (int j = 0; j < n_kt; ++j) {
      const int u = j & 1;
      const uint2 bits = bits_next;
      if (valid_q && j + 1 < n_kt) bits_next = __ldg(reinterpret_cast<const uint2*>(mrow + 2 * (j + 1)));
      if (!(ok = mbar_wait(s_full(u), (j >> 1) & 1, abort_flag, p.err))) break;
      tc_fence_after();
      uint32_t sv[64];
      {
        uint32_t a[32], c[32];
        tmem_ld32(tmem + lane_base + C::S_COL + u * 64, a);
        tmem_ld32(tmem + lane_base + C::S_COL + u * 64 + 32, c);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          sv[i] = a[i];
          sv[32 + i] = c[i];
        }
      }
      tc_fence_before();
      mbar_arrive(s_free(u));
      // the maximum over all 64 keys (both threads of the row find the same),
      // the exponentials for this thread's 32
      // of the raw selected scores, scaled once: the scale is positive, so
      // max(s) * scale = max(s * scale) under rounding as well.  The reference
      // moves only when a selected score passes it by 2^8, which the maximum
      // over all 64 keys bounds: the selection is consulted only when that
      // passes (the first tiles of a row, or an unselected key far above it).
      float ur = neg_inf();
#pragma unroll
      for (int c = 0; c < 64; ++c) ur = fmaxf(ur, __uint_as_float(sv[c]));
      float mt = ur * p.scale_log2;
      if (mt > m_ref + 8.f) {
        float mr = neg_inf();
#pragma unroll
        for (int c = 0; c < 64; ++c)
          mr = fmaxf(mr, ((c < 32 ? bits.x : bits.y) & (1u << (c & 31))) ? __uint_as_float(sv[c]) : neg_inf());
        mt = mr * p.scale_log2;
      }
      const uint32_t mine = hf ? bits.y : bits.x;
      // the reference moves when a score passes it by more than 2^8; O and l
      // follow it (TMEM loads and stores are warp-wide: a row that keeps its
      // reference is scaled by 1).  Rescaling O needs the previous P.V done.
      const bool move = mt > m_ref + 8.f;
      // O holds something once any earlier key of the row was selected (the
      // reference is finite then), whichever half of the tile it was in
      const bool need = move && j > 0 && m_ref != neg_inf();
      const float f = need ? ex2_approx(m_ref - mt) : 1.f;
      const bool rescaled = __any_sync(0xffffffffu, need);
      if (rescaled) {
        if (!(ok = mbar_wait(pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag, p.err))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = hf * 128; c0 < hf * 128 + 128; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(tmem + lane_base + c0, o);
        }
      }
      l *= f;
      if (move) m_ref = mt;
      uint32_t pk[16];
      float lsum = 0.f;
      // p = 2^(s * scale - m_ref) for this thread's selected keys, one FMA each
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const float s0 = __uint_as_float(hf ? sv[32 + c] : sv[c]), s1 = __uint_as_float(hf ? sv[33 + c] : sv[c + 1]);
        const float p0 = (mine & (1u << c)) ? ex2_approx(fmaf(s0, p.scale_log2, -m_ref)) : 0.f;
        const float p1 = (mine & (1u << (c + 1))) ? ex2_approx(fmaf(s1, p.scale_log2, -m_ref)) : 0.f;
        const uint32_t w = pack_bf16x2(p0, p1);
        lsum += bf16lo_to_f32(w) + bf16hi_to_f32(w);
        pk[c >> 1] = w;
      }
      l += lsum;
      // P buffer u (tensor memory) was last read by the P.V of tile j - 2
      if (j >= 2 && !(ok = mbar_wait(pv_done(u), ((j >> 1) - 1) & 1, abort_flag, p.err))) break;
      tc_fence_after();
      tmem_st16(tmem + lane_base + C::P_COL + u * 32 + hf * 16, pk);  // this thread's 32 keys of the row
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full(u));
    }
    if (ok && n_kt > 0) ok = mbar_wait(pv_done((n_kt - 1) & 1), ((n_kt - 1) >> 1) & 1, abort_flag, p.err);
    tc_fence_after();
    // the row sum is the two threads' halves: exchanged through the (now idle) value stages
    float* lx = reinterpret_cast<float*>(smem + C::OFF_V);
    lx[hf * 128 + row] = l;
    named_bar_sync(1, 256);
    const float l_row = lx[row] + lx[128 + row];
    const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
    const int64_t orow = (int64_t)t * p.H + h;
#pragma unroll 1
    for (int c0 = hf * 128; c0 < hf * 128 + 128; c0 += 32) {
      uint32_t o[32];
      if (n_kt > 0) {
        tmem_ld32(tmem + lane_base + c0, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (valid_q && ok) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kHead + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * i]) * inv, __uint_as_float(o[8 * i + 1]) * inv),
                              pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv),
                              pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv),
                              pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv));
      }
    }
    if (hf == 0 && valid_q && ok && p.lse != nullptr)
      p.lse[orow] = l_row > 0.f ? (m_ref + lg2_approx(l_row)) * 0.69314718055994531f : neg_inf();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

cudaError_t launch_with(const void* kern, dim3 grid, int block, size_t smem, void** args, cudaStream_t stream,
                        bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at = pdl_attribute();
  cfg.attrs = &at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, kern, args);
}

template <int N, bool KEYS>
cudaError_t launch_project_one(const MhaProjectLaunch& a, const void* w, __nv_bfloat16* out, cudaStream_t stream) {
  using C = ProjCfg<N>;
  CUtensorMap tm_c, tm_w;
  {
    const uint64_t dims[2] = {(uint64_t)(kLatent + kRope), (uint64_t)a.rows};
    const uint64_t strides[1] = {(uint64_t)a.c_stride * 2};
    const uint32_t box[2] = {64, 128};
    if (encode_tmap(&tm_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.c, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)kLatent, (uint64_t)a.H * N};
    const uint64_t strides[1] = {(uint64_t)kLatent * 2};
    const uint32_t box[2] = {64, (uint32_t)N};
    if (encode_tmap(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  ProjParams p;
  p.c = static_cast<const __nv_bfloat16*>(a.c);
  p.c_stride = a.c_stride;
  p.rows = a.rows;
  p.H = a.H;
  p.out = out;
  p.err = a.err;
  auto kern = mha_project_kernel<N, KEYS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  void* args[] = {&tm_c, &tm_w, &p};
  const int64_t n_tiles = (a.rows + 127) / 128 * a.H;
  const dim3 grid((unsigned)std::min<int64_t>(n_tiles, a.num_sms), 1, 1);
  return launch_with(reinterpret_cast<const void*>(kern), grid, C::THREADS, C::SMEM_BYTES, args, stream, true);
}

}  // namespace

cudaError_t launch_mha_project(const MhaProjectLaunch& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  cudaError_t e = launch_project_one<kHead - kRope, true>(a, a.w_uk, static_cast<__nv_bfloat16*>(a.k_out), stream);
  if (e != cudaSuccess) return e;
  return launch_project_one<kHead, false>(a, a.w_uv, static_cast<__nv_bfloat16*>(a.v_out), stream);
}

int mha_mask_words(int max_seqlen_k) { return ((max_seqlen_k + 31) / 32 + 1) / 2 * 2; }

cudaError_t launch_mha_attend(const MhaAttendLaunch& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  // (1) selection masks
  MaskParams mp;
  mp.idx = a.idx;
  mp.ld_idx = a.ld_idx;
  mp.k = a.k_sel;
  mp.T = a.T;
  mp.W = a.W;
  mp.q_n = a.plan.q_n;
  mp.mask = a.mask;
  mp.err = a.err;
  {
    void* args[] = {&mp};
    const size_t smem = (size_t)a.W * 4;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(mha_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_with(reinterpret_cast<const void*>(mha_mask_kernel), dim3(a.T, 1, 1), 256, smem, args,
                                stream, true);
    if (e != cudaSuccess) return e;
  }
  // (2) attention
  CUtensorMap tm_q, tm_k, tm_v;
  {
    const uint64_t dims[3] = {(uint64_t)kHead, (uint64_t)a.H, (uint64_t)a.T};
    const uint64_t strides[2] = {(uint64_t)kHead * 2, (uint64_t)kHead * a.H * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (encode_tmap(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const CacheView* views[2] = {&a.k, &a.v};
  CUtensorMap* maps[2] = {&tm_k, &tm_v};
  for (int i = 0; i < 2; ++i) {
    const uint64_t dims[3] = {(uint64_t)kHead, (uint64_t)a.H, (uint64_t)views[i]->num_rows};
    const uint64_t strides[2] = {(uint64_t)kHead * 2, (uint64_t)views[i]->row_stride * 2};
    const uint32_t box[3] = {64, 1, 64};
    if (encode_tmap(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, views[i]->base, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  AttParams p;
  p.plan = a.plan;
  p.kv = a.k;
  p.mask = a.mask;
  p.W = a.W;
  p.H = a.H;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.err = a.err;
  cudaError_t e = cudaFuncSetAttribute(mha_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       AttCfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  void* args[] = {&tm_q, &tm_k, &tm_v, &p};
  const dim3 grid((unsigned)a.max_groups, (unsigned)a.H, 1);
  return launch_with(reinterpret_cast<const void*>(mha_attend_kernel), grid, AttCfg::THREADS, AttCfg::SMEM_BYTES,
                     args, stream, true);
}

}  // namespace dsa

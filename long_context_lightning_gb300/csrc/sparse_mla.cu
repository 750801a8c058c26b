// sparse_mla.cu -- sparse MLA in MQA mode over the selected latent rows.
//
// For query t and head h, over the selected positions s:
//   z_s = scale * Q[t, h, :D] . C[s, :D],  p = softmax(z),
//   O[t, h, :] = sum_s p_s C[s, :D_v],  LSE[t, h] = log sum_s exp(z_s)
// ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works /
// Model, sparse-MLA bullet: sparse MLA in MQA mode over the top-k tokens, all
// heads sharing the one latent row of a token).
//
// Row gather.  The selected rows of a query are taken 128 at a time into one
// tile of shared memory, D/64 column blocks of [128 rows x 64 dims] (128-byte
// swizzle), by TMA tile::gather4 (four rows x 64 dims per instruction).  A
// gather4 costs its warp ~30 ns (lanes in series), so the copies are spread:
// gather warp w owns the column blocks w and w+4, and the last block (it holds
// P^T during the PV, so it is freed last) is gathered by the eight softmax
// warps, idle at that point.  Each column block is refilled as soon as the PV
// MMAs that read it complete, so the next tile's copies overlap the end of
// this tile's PV; and once a tile has landed, the next tile's rows are
// bulk-prefetched into L2 (HBM is otherwise idle while a tile is consumed), so
// those copies read L2.
//
// Tensor cores.  The same tile serves two MMAs:
//   S^T[key, h] = C[key, :] . Q[h, :]^T     M = 128 keys, N = 64 heads, K = D
//   O^T[v, h]  += C[key, v]^T . P^T[key, h] M = 128 value dims per block, N = 64
//                 heads, K = 128 keys (C read MN-major, P^T MN-major)
// so the 64-head MQA tile is a real dense contraction with every TMEM lane in
// use (O^T: D_v/128 x 64 columns, S^T: 64 columns).  Each product is issued as
// one unbroken run of MMAs once its operands are complete: waits or other
// control work between MMAs leave the tensor pipe idle.  P^T is written into
// the tile's rope block, dead once S^T has been formed.
//
// Softmax.  One thread owns one key for 32 heads.  Probabilities are taken
// against a per-head reference m that only moves when some score passes it
// by more than 2^16 (the first tile always moves it): the exact result does
// not depend on m, P in bf16 keeps its relative precision at any magnitude,
// and fp32 sums stay far from overflow.  The common tile therefore needs no
// max reduction at all, only one barrier that ORs the overflow test.
//
// Split over a cluster: the selected rows of one query are divided among the
// blocks of a thread-block cluster; each block keeps its partial (m, l, O).
// Combine: every block writes its unnormalised partial O^T as bf16 rows
// [head pair][value dim] with its (m, l) per head in front, one slab per owner
// of a value slice; once the owner reports its tile memory free, the slab
// moves there with one bulk copy (shared::cta -> shared::cluster), and the
// owner weights and sums the slabs of its slice.  One exchange, no global
// traffic.
//
// Warp roles (416 threads, one block per SM):
//   warps 0..3   row gather (index -> pool row, paged or contiguous) of the
//                column blocks before the last; next tile's L2 prefetch
//   warp 4       TMEM owner, query TMA, MMA issuer (one thread)
//   warps 5..12  softmax: two warps per TMEM lane quadrant, 32 heads each;
//                the last column block's gather; then the combine
#include <algorithm>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 16.0f;  // move the reference only past 2^16
constexpr int kSoftmaxThreads = 256;
constexpr int kProducerThreads = 128;
constexpr int kMaxSplit = 8;          // blocks per cluster (splits of one query's rows)
constexpr int kRows = 128;            // selected rows per tile
constexpr int kBlk = kRows * 128;     // one [128 rows x 64 dims] bf16 block
constexpr int kSlabHeader = 512;      // (m, l) x 64 heads, fp32

template <int NB, int MB>
struct MlaCfg {
  static constexpr int THREADS = kProducerThreads + 32 + kSoftmaxThreads;
  static constexpr int STAGE = NB * kBlk;                 // one tile of gathered rows
  static constexpr int OFF_Q = 0;                         // NB x [64 heads x 64 dims]
  static constexpr int OFF_KV = OFF_Q + NB * 64 * 128;    // NB blocks of [128 rows x 64 dims]
  static constexpr int OFF_VALID = OFF_KV + STAGE;        // 128 int
  static constexpr int OFF_RED = OFF_VALID + kRows * 4;      // 4 x 64 float
  static constexpr int OFF_MREF = OFF_RED + 4 * 64 * 4;      // 64 float
  static constexpr int OFF_ALPHA = OFF_MREF + 64 * 4;        // 64 float
  static constexpr int OFF_F = OFF_ALPHA + 64 * 4;           // kMaxSplit x 64 float
  static constexpr int OFF_BAR = OFF_F + kMaxSplit * 64 * 4;
  static constexpr int N_BARS = NB + 10;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int OFF_LAYER = OFF_MISC + 16;          // output, LSE, heads of this block's layer
  static constexpr int SMEM_BYTES = OFF_LAYER + 32 + 1024;
  static constexpr int S_COL = MB * 64;                   // O^T in columns [0, S_COL), then S^T
  static constexpr int TMEM_COLS = (S_COL + 64) <= 256 ? 256 : 512;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct LayerOut {
  __nv_bfloat16* out;
  float* lse;
  int32_t H;
  int32_t d_v;
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
  int32_t plan_early;
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

// Bounded wait with cluster-scope acquire (remote arrivals and copies).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, int* err_word) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err_word, DEV_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

template <int NB, int MB>
__global__ void __launch_bounds__(kProducerThreads + 32 + kSoftmaxThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
                      const __grid_constant__ CUtensorMap tm_q2, const __grid_constant__ CUtensorMap tm_q3,
                      const __grid_constant__ CUtensorMap tm_c0, const __grid_constant__ CUtensorMap tm_c1,
                      const __grid_constant__ CUtensorMap tm_c2, const __grid_constant__ CUtensorMap tm_c3,
                      MlaParams p) {
  using C = MlaCfg<NB, MB>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  int* valid_s = reinterpret_cast<int*>(smem + C::OFF_VALID);
  float* red_s = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* mref_s = reinterpret_cast<float*>(smem + C::OFF_MREF);
  float* alpha_s = reinterpret_cast<float*>(smem + C::OFF_ALPHA);
  float* f_s = reinterpret_cast<float*>(smem + C::OFF_F);  // [source block][head]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  // one phase per tile each: column blocks [0, NB_A) / [NB_A, NB) of the tile
  // landed (bytes); column block kb read by every MMA of the tile (commit);
  // S^T formed (commit); P^T written (softmax threads); the tile's valid flags
  // written (gather warp 0)
  constexpr int NB_A = (NB + 1) / 2;  // blocks of the first S^T run
  auto bar_full = [&](int part) { return smem_u32(bars + part); };
  auto bar_empty = [&](int kb) { return smem_u32(bars + 2 + kb); };
  const uint32_t bar_s_full = smem_u32(bars + NB + 2);
  const uint32_t bar_p_full = smem_u32(bars + NB + 3);
  const uint32_t bar_valid = smem_u32(bars + NB + 4);
  const uint32_t bar_q_full = smem_u32(bars + NB + 5);
  const uint32_t bar_o_done = smem_u32(bars + NB + 6);
  const uint32_t bar_drain = smem_u32(bars + NB + 7);
  const uint32_t bar_recv = smem_u32(bars + NB + 8);   // peers' slabs landed (bytes)
  const uint32_t bar_ready = smem_u32(bars + NB + 9);  // peers' tile memory free (remote arrivals)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const int t = blockIdx.y % p.T;
  const int li = blockIdx.y / p.T;
  const MlaLayerView& L = p.layer[li];
  const CUtensorMap* tm_q = li == 0 ? &tm_q0 : li == 1 ? &tm_q1 : li == 2 ? &tm_q2 : &tm_q3;
  const CUtensorMap* tm_c = li == 0 ? &tm_c0 : li == 1 ? &tm_c1 : li == 2 ? &tm_c2 : &tm_c3;
  const int slice = p.d_v / (int)csize;  // value dims owned by each block of the cluster
  // a slab: header, then [32 head pairs][slice value dims] words (bf16 pairs)
  const uint32_t slab_bytes = (uint32_t)(kSlabHeader + slice * 32 * 4);
  const int ls = __ffs(slice) - 1;  // slice is a power of two (d_v and the cluster size are)

  if (threadIdx.x == 0) {
    mbar_init(bar_full(0), 1);
    mbar_init(bar_full(1), 1);
    for (int kb = 0; kb < NB; ++kb) mbar_init(bar_empty(kb), 1);
    mbar_init(bar_valid, 32);
    mbar_init(bar_s_full, 1);
    mbar_init(bar_p_full, kSoftmaxThreads);
    mbar_init(bar_q_full, 1);
    mbar_init(bar_o_done, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_recv, 1);
    mbar_init(bar_ready, csize > 1 ? csize - 1 : 1);
    *abort_flag = 0;
    // the combine reads these from shared memory rather than from the
    // parameter bank (indexed by layer at run time)
    LayerOut* lo = reinterpret_cast<LayerOut*>(smem + C::OFF_LAYER);
    lo->out = L.out;
    lo->lse = L.lse;
    lo->H = L.H;
    lo->d_v = p.d_v;
    fence_mbar_init();
    prefetch_tmap(tm_c);
    // the peers' slabs are counted in bytes; this arrival opens the phase
    if (csize > 1) mbar_arrive_expect_tx(bar_recv, (csize - 1) * slab_bytes);
  }
  if (threadIdx.x >= 160 && threadIdx.x < 224) mref_s[threadIdx.x - 160] = -INFINITY;
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // remote arrivals and copies may target this block's barriers from here on
  if (csize > 1) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the query is a caller input: its load may overlap the previous grid
  if (warp == 4 && lane == 0) {
    mbar_arrive_expect_tx(bar_q_full, NB * 64 * 128);
    for (int kb = 0; kb < NB; ++kb) tma_load_3d(sbase + C::OFF_Q + kb * 64 * 128, tm_q, bar_q_full, kb * 64, 0, t);
  }
  int my_tiles = 0;
  // ------------------------------------------------ the tiles of this block
  auto run_tiles = [&]() {
    // The plan is read before the wait when it was written two or more grids
    // back (complete before this grid could start); L2 loads, no stale L1.
    // The sequence's first pool row of a contiguous cache is a caller input.
    int n_t = 0, b = 0;
    int64_t seq_base = 0;
    auto read_plan = [&]() {
      n_t = __ldcg(p.q_n + t);
      b = __ldcg(p.q_seq + t);
      if (!L.kv.paged && !L.kv.rows && b >= 0) seq_base = __ldg(L.kv.seq_start + b);
    };
    if (p.plan_early) read_plan();
    pdl_wait();  // positions and plan of the previous grids are complete from here on
    pdl_trigger();
    if (!p.plan_early) read_plan();

    const int nvalid = min(n_t, p.k);
    const int tiles = (nvalid + kRows - 1) / kRows;
    const int j0 = (int)((int64_t)tiles * crank / csize), j1 = (int)((int64_t)tiles * (crank + 1) / csize);
    my_tiles = j1 - j0;

    // Lane l of a gathering warp resolves rows 4l..4l+3 of a tile to pool rows.
    const int32_t* idx_row = p.idx + (int64_t)t * p.ld_idx;
    int32_t r4[4];
    bool v4[4];
    auto resolve = [&](int jj) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = (j0 + jj) * kRows + 4 * lane + k;
        int pos = e < nvalid ? __ldg(idx_row + e) : -1;
        // a position is a token of the sequence, or a pool row for a cache of rows
        if ((!L.kv.rows && pos >= n_t) || pos < -1) {
          if (warp == 0) atomicOr(p.err, DEV_ERR_BAD_INDEX);
          pos = -1;
        }
        int64_t row = -1;
        if (pos >= 0) {
          if (L.kv.paged || L.kv.rows) {
            row = cache_row(L.kv, b, pos);
          } else {
            row = seq_base + pos;
            if (row < 0 || row >= L.kv.num_rows) row = -1;
          }
          if (row < 0 && warp == 0) atomicOr(p.err, DEV_ERR_BAD_INDEX);
        }
        v4[k] = row >= 0;
        r4[k] = row >= 0 ? (int32_t)row : 0;  // an unused slot reads pool row 0 (finite data; weight 0)
      }
    };
    // Column block NB-1 (it holds P^T while the PV runs, so it is released
    // last) is gathered by the softmax warps, idle at that point: lanes
    // 4j..4j+3 of softmax warp j, four copies per warp rather than one warp's
    // thirty-two.
    auto gather_last_block = [&]() {
      if ((lane >> 2) == warp - 5)
        tma_gather4(sbase + C::OFF_KV + lane * 512 + (NB - 1) * kBlk, tm_c, bar_full(1), (NB - 1) * 64, r4[0], r4[1], r4[2],
                    r4[3]);
    };

    if (warp < 4) {
      // ------------------------------------------------------------ row gather
      // Warp w owns the column blocks kb = w, w+4 < NB-1 of every tile and
      // gathers its lanes' rows for each of them.  A block is refilled as soon
      // as the PV that reads it has completed; S^T waits for the whole tile.
      bool bad = false;
      if (my_tiles > 0) resolve(0);
      for (int jj = 0; jj < my_tiles; ++jj) {
        const uint32_t par = (jj & 1) ^ 1;  // phase of the previous tile
        const uint32_t dst = sbase + C::OFF_KV + lane * 512;
        for (int kb = warp; kb < NB - 1; kb += 4) {
          bad |= !mbar_wait(bar_empty(kb), par, abort_flag, p.err);
          if (kb == 0) {
            // block 0 is released by the first MMA group of the previous PV,
            // issued after that tile's softmax had read these flags
#pragma unroll
            for (int k = 0; k < 4; ++k) valid_s[4 * lane + k] = v4[k];
            mbar_arrive(bar_valid);
            // one arrival with each part's bytes opens its phase; blocks of other
            // warps may land before it (the count goes negative).  Block 0 is
            // released after the previous S^T, so both previous phases are done.
            if (lane == 0) {
              mbar_arrive_expect_tx(bar_full(0), NB_A * kBlk);
              mbar_arrive_expect_tx(bar_full(1), (NB - NB_A) * kBlk);
            }
          }
          __syncwarp();
          const uint32_t bar = bar_full(kb < NB_A ? 0 : 1);
          if (!bad) tma_gather4(dst + kb * kBlk, tm_c, bar, kb * 64, r4[0], r4[1], r4[2], r4[3]);
        }
        if (jj + 1 < my_tiles) {
          // Shared memory holds one tile.  Once this tile has landed, HBM is idle
          // while it is consumed: the next tile's rows stream into L2 then, and
          // its gathers read L2.  The four warps split the rows (lane l, warp w:
          // row 4l + w), one bulk prefetch of a whole row each.
          resolve(jj + 1);
          int32_t rp = r4[0];
          bool vp = v4[0];
#pragma unroll
          for (int k = 1; k < 4; ++k)
            if (warp == k) { rp = r4[k]; vp = v4[k]; }
          if (!bad) bad = !mbar_wait(bar_full(1), jj & 1, abort_flag, p.err);
          if (!bad && vp) prefetch_l2_bulk(L.kv.base + (int64_t)rp * L.kv.row_stride, (uint32_t)p.d_qk * 2u);
        }
      }
    } else if (warp == 4) {
      // ---------------------------------------------- query TMA + MMA issuer
      if (lane == 0) {
        bool bad = !mbar_wait(bar_q_full, 0, abort_flag, p.err);
        if (bad) mbar_wait_drain(bar_q_full, 0);  // the query copy lands before the block may exit
        constexpr uint32_t idesc_s = mma_idesc_bf16(128, 64, false, false);
        constexpr uint32_t idesc_o = mma_idesc_bf16(128, 64, true, true);
        // descriptors of block 0 of each operand; a block or K step moves the
        // start address field (address >> 4, no carry out of its 14 bits)
        const uint64_t dq = smem_desc_sw128(sbase + C::OFF_Q, 16, 1024);
        const uint64_t dk = smem_desc_sw128(sbase + C::OFF_KV, 16, 1024);
        const uint64_t dv = smem_desc_sw128(sbase + C::OFF_KV, kBlk, 1024);
        const uint64_t dp = dv + (uint64_t)(((NB - 1) * kBlk) >> 4);
        // Each product is one unbroken run of MMAs: control work between them
        // starves the tensor pipe.  The tile was written by TMA and its mbarrier
        // orders it for the tensor cores.
        for (int jj = 0; jj < my_tiles && !bad; ++jj) {
          const uint32_t par = jj & 1;
          // S^T = C . Q^T over all D/64 column blocks, in two runs: the blocks
          // released first by the previous PV land first
          if (!mbar_wait(bar_full(0), par, abort_flag, p.err)) { bad = true; break; }
#pragma unroll
          for (int kb = 0; kb < NB_A; ++kb)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(tmem + C::S_COL, dk + (uint64_t)((kb * kBlk + kk * 32) >> 4),
                       dq + (uint64_t)((kb * 64 * 128 + kk * 32) >> 4), idesc_s, (kb | kk) != 0);
          if (!mbar_wait(bar_full(1), par, abort_flag, p.err)) { bad = true; break; }
#pragma unroll
          for (int kb = NB_A; kb < NB; ++kb)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(tmem + C::S_COL, dk + (uint64_t)((kb * kBlk + kk * 32) >> 4),
                       dq + (uint64_t)((kb * 64 * 128 + kk * 32) >> 4), idesc_s, 1u);
          mma_commit(bar_s_full);
          // O^T += C^T . P^T over the tile's 128 keys; each column block is
          // released to the gather as soon as the MMAs reading it complete
          if (!mbar_wait(bar_p_full, par, abort_flag, p.err)) { bad = true; break; }
          tc_fence_after();
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16(tmem + mb * 64, dv + (uint64_t)((2 * mb * kBlk + kk * 2048) >> 4),
                       dp + (uint64_t)((kk * 2048) >> 4), idesc_o, (jj | kk) != 0);
            if (2 * mb < NB - 1) mma_commit(bar_empty(2 * mb));
            if (2 * mb + 1 < NB - 1) mma_commit(bar_empty(2 * mb + 1));
          }
          mma_commit(bar_empty(NB - 1));  // the P^T block, read by every PV above
        }
        mma_commit(bar_o_done);
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0);
      }
    } else {
      // ------------------------------------------------------------- softmax
      const int quad = warp & 3;
      const int half = (warp - 5) >> 2;   // heads 32*half .. +31
      const int st = threadIdx.x - 160;   // 0..255
      const int h0 = half * 32;
      const int srow = quad * 32 + lane;  // key of S^T held by this lane
      const float c = L.scale * kLog2e;
      const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
      if (my_tiles > 0) {
        resolve(0);
        gather_last_block();
      }
      float lsum[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) lsum[i] = 0.f;
      bool bad = false;
      for (int jj = 0; jj < my_tiles; ++jj) {
        const uint32_t par = jj & 1;
        bad |= !mbar_wait(bar_valid, par, abort_flag, p.err);
        bad |= !mbar_wait(bar_s_full, par, abort_flag, p.err);
        tc_fence_after();
        const bool kv = valid_s[srow] != 0;
        uint32_t r[32];  // this key's raw scores for heads h0..h0+31
        auto load_scores = [&]() {
          tmem_ld32(lane_base + C::S_COL + h0, r);
          tmem_wait_ld();
        };
        // d = score x scale - the head's reference (log2 units), one FMA each:
        // it decides the overflow vote and gives the probability 2^d
        float d[32];
        auto diffs = [&]() {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mref_s + h0 + i);
            d[i] = fmaf(__uint_as_float(r[i]), c, -m4.x);
            d[i + 1] = fmaf(__uint_as_float(r[i + 1]), c, -m4.y);
            d[i + 2] = fmaf(__uint_as_float(r[i + 2]), c, -m4.z);
            d[i + 3] = fmaf(__uint_as_float(r[i + 3]), c, -m4.w);
          }
        };
        load_scores();
        diffs();
        bool over = false;
#pragma unroll
        for (int i = 0; i < 32; ++i) over |= d[i] > kRescaleLog2;
        if (bar_red_or(4, kSoftmaxThreads, kv && over)) {
          // move the reference of every head whose tile max passed it
          {
            float x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = kv ? __uint_as_float(r[i]) * c : -INFINITY;
            red_s[quad * 64 + h0 + lane] = transpose_reduce32<true>(x, lane);
          }
          named_bar_sync(3, kSoftmaxThreads);
          bool rescale = false;
          if (st < 64) {
            const float mt = fmaxf(fmaxf(red_s[st], red_s[64 + st]), fmaxf(red_s[128 + st], red_s[192 + st]));
            const float mr = mref_s[st];
            float alpha = 1.f;
            if (mt > mr + kRescaleLog2 || (mr == -INFINITY && mt > -INFINITY)) {
              alpha = (mr == -INFINITY) ? 0.f : ex2_approx(mr - mt);
              mref_s[st] = mt;
              rescale = mr != -INFINITY;
            }
            alpha_s[st] = alpha;
          }
          if (bar_red_or(4, kSoftmaxThreads, rescale)) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 a4 = *reinterpret_cast<const float4*>(alpha_s + h0 + i);
              lsum[i] *= a4.x; lsum[i + 1] *= a4.y; lsum[i + 2] *= a4.z; lsum[i + 3] *= a4.w;
            }
            // O^T holds every earlier tile once the PV of tile jj-1 completed (the
            // PV of jj-2 completed before this tile's blocks could be gathered)
            if (jj > 0) bad |= !mbar_wait(bar_empty(NB - 1), (jj - 1) & 1, abort_flag, p.err);
            tc_fence_after();
            if (!__any_sync(0xffffffffu, bad)) {  // warp-uniform: tcgen05.ld/st are .aligned
#pragma unroll 1
              for (int q = 0; q < 2 * MB; ++q) {  // 16 columns at a time keeps the registers low
                const uint32_t col = lane_base + (q >> 1) * 64 + h0 + (q & 1) * 16;
                const float* a = alpha_s + h0 + (q & 1) * 16;
                uint32_t o[16];
                tmem_ld16(col, o);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a[i]);
                tmem_st16(col, o);
              }
              tmem_wait_st();
            }
          }
          load_scores();  // reloaded rather than kept live across the rescale
          diffs();        // against the moved references
        }
        // probabilities, running sums, this key's P^T row for heads h0..h0+31 (bf16)
        const uint32_t prow = sbase + C::OFF_KV + (NB - 1) * kBlk + srow * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float pv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = cc * 8 + j;
            pv[j] = kv ? ex2_approx(d[i]) : 0.f;
            lsum[i] += pv[j];
          }
          const int chunk = half * 4 + cc;
          st_shared_v4(prow + ((chunk ^ (srow & 7)) << 4), pack_bf16x2(pv[0], pv[1]), pack_bf16x2(pv[2], pv[3]),
                       pack_bf16x2(pv[4], pv[5]), pack_bf16x2(pv[6], pv[7]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar_p_full);
        if (jj + 1 < my_tiles) {
          // the next tile's block NB-1 replaces this P^T once the PV has read it
          resolve(jj + 1);
          bad |= !mbar_wait(bar_empty(NB - 1), jj & 1, abort_flag, p.err);
          if (!bad) gather_last_block();
        }
      }
      // l per head over this block's keys
      red_s[quad * 64 + h0 + lane] = transpose_reduce32<false>(lsum, lane);
      named_bar_sync(3, kSoftmaxThreads);
      if (my_tiles > 0) bad |= !mbar_wait(bar_o_done, 0, abort_flag, p.err);
      tc_fence_after();
    }
  };

  auto combine = [&]() {
    // ------------------------------------------------- combine over the cluster
    // Every role is past its loop: this block's stages are free for the slabs.
    // recv: [source block][slab], send: [owner block][slab]; a slab is the
    // source's (m, l) per head, then one row per head pair of the owner's
    // slice of value dims, each word the pair as two bf16.
    __syncthreads();
    const LayerOut lo = *reinterpret_cast<const LayerOut*>(smem + C::OFF_LAYER);
    uint8_t* recv = smem + C::OFF_KV;
    uint8_t* send = recv + csize * slab_bytes;
    if (threadIdx.x == 0)
      for (uint32_t o = 0; o < csize; ++o)
        if (o != crank) mbar_arrive_remote(dsmem_addr(bar_ready, o));
    if (warp >= 5) {
      const int quad = warp & 3;
      const int h0 = ((warp - 5) >> 2) * 32;
      const int st = threadIdx.x - 160;
      const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
      if (st < 64) {
        const float m_own = mref_s[st];
        const float l_own = red_s[st] + red_s[64 + st] + red_s[128 + st] + red_s[192 + st];
        for (uint32_t o = 0; o < csize; ++o) {
          float* hdr = reinterpret_cast<float*>(o == crank ? recv + crank * slab_bytes : send + o * slab_bytes);
          hdr[st] = m_own;
          hdr[64 + st] = l_own;
        }
      }
      // one-shot code: kept a loop, since every unrolled copy would be a fresh
      // instruction fetch
#pragma unroll 1
      for (int mb = 0; mb < MB; ++mb) {
        const int vq = mb * 128 + quad * 32;  // this warp's first value dim (warp-uniform)
        if (vq >= lo.d_v) continue;
        uint32_t r[32];
        if (my_tiles > 0) {
          tmem_ld32(lane_base + mb * 64 + h0, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        const int owner = vq >> ls;  // a slice holds whole warps (>= 32 dims)
        const int v = vq - (owner << ls) + lane;
        uint8_t* slab = owner == (int)crank ? recv + crank * slab_bytes : send + owner * slab_bytes;
        // lane = value dim: a warp writes 32 consecutive words of each head-pair row
        uint32_t* col = reinterpret_cast<uint32_t*>(slab + kSlabHeader) + (h0 / 2) * slice + v;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          col[i * slice] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
      }
      fence_proxy_async_smem();  // the slabs are read by the bulk-copy engine
      named_bar_sync(3, kSoftmaxThreads);
      if (st == 0 && csize > 1) {
        // a peer's stages may be overwritten only after its own loop has ended
        if (mbar_wait_cluster(bar_ready, 0, p.err)) {
          for (uint32_t o = 0; o < csize; ++o) {
            if (o == crank) continue;
            bulk_copy_smem_to_peer(dsmem_addr(smem_u32(recv + crank * slab_bytes), o), smem_u32(send + o * slab_bytes),
                                   slab_bytes, dsmem_addr(bar_recv, o));
          }
        }
      }
      bool ok = true;
      if (csize > 1) ok = mbar_wait_cluster(bar_recv, 0, p.err);  // every source's slab has landed
      // every peer's copy out of its staging area has completed: a peer may
      // leave once all blocks have passed this point (the wait is at the end)
      if (csize > 1) cluster_arrive();
      // weight of each source per head: four threads per head, each with the
      // sources sub and sub + 4; max and sum over a head's sources by shuffles
      {
        const int h = st >> 2, sub = st & 3;
        const float* h0p = reinterpret_cast<const float*>(recv + sub * slab_bytes);
        const float* h1p = reinterpret_cast<const float*>(recv + (sub + 4) * slab_bytes);
        const bool has0 = sub < (int)csize, has1 = sub + 4 < (int)csize;
        const float m0 = has0 ? h0p[h] : -INFINITY, m1 = has1 ? h1p[h] : -INFINITY;
        const float l0 = has0 ? h0p[64 + h] : 0.f, l1 = has1 ? h1p[64 + h] : 0.f;
        float M = fmaxf(m0, m1);
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
        const float e0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - M), e1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - M);
        float Lsum = l0 * e0 + l1 * e1;
        Lsum += __shfl_xor_sync(0xffffffffu, Lsum, 1);
        Lsum += __shfl_xor_sync(0xffffffffu, Lsum, 2);
        const float inv = (ok && Lsum > 0.f) ? rcp_approx(Lsum) : 0.f;
        if (has0) f_s[sub * 64 + h] = e0 * inv;
        if (has1) f_s[(sub + 4) * 64 + h] = e1 * inv;
        if (sub == 0 && crank == 0 && lo.lse != nullptr && h < lo.H)
          lo.lse[(int64_t)t * lo.H + h] = Lsum > 0.f ? (M + lg2_approx(Lsum)) * kLn2 : -INFINITY;
      }
      named_bar_sync(3, kSoftmaxThreads);
      // this block's value slice of every head: a thread takes one head pair and
      // four consecutive value dims per item (one 16-byte load per source, one
      // 8-byte store per head); a warp's items are contiguous in every slab
      const int v0 = (int)crank * slice;
      const int lvg = ls - 2;
      const int items = 32 << lvg;
      const float2* fw = reinterpret_cast<const float2*>(f_s);  // [source][head pair]
      for (int it = st; it < items; it += kSoftmaxThreads) {
        const int hp = it >> lvg;
        const int vg = it & ((1 << lvg) - 1);
        const int h = 2 * hp;
        if (h >= lo.H) continue;
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < kMaxSplit; ++r) {
          if (r < (int)csize) {
            const uint4 w = *reinterpret_cast<const uint4*>(recv + r * slab_bytes + kSlabHeader +
                                                             (size_t)(hp * slice + 4 * vg) * 4);
            const float2 f2 = fw[r * 32 + hp];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              a0[j] = fmaf(f2.x, bf16lo_to_f32(ws[j]), a0[j]);
              a1[j] = fmaf(f2.y, bf16hi_to_f32(ws[j]), a1[j]);
            }
          }
        }
        __nv_bfloat16* o0 = lo.out + ((int64_t)t * lo.H + h) * lo.d_v + v0 + 4 * vg;
        *reinterpret_cast<uint2*>(o0) = make_uint2(pack_bf16x2(a0[0], a0[1]), pack_bf16x2(a0[2], a0[3]));
        if (h + 1 < lo.H)
          *reinterpret_cast<uint2*>(o0 + lo.d_v) = make_uint2(pack_bf16x2(a1[0], a1[1]), pack_bf16x2(a1[2], a1[3]));
      }
    }
  };

  run_tiles();
  combine();
  // no block may leave while a peer's copy could still read its staging area
  // (the softmax warps arrived after their slabs landed, the others here)
  if (csize > 1) {
    if (warp < 5) cluster_arrive();
    cluster_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int NB, int MB>
cudaError_t launch_t(const MlaLaunch& a, cudaStream_t stream, int which) {
  using C = MlaCfg<NB, MB>;
  auto kern = sparse_mla_kernel<NB, MB>;
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
    {  // latent pool rows for tile::gather4: box of 64 dims x one row
      const uint64_t dims[2] = {(uint64_t)a.d_qk, (uint64_t)lv.kv.num_rows};
      const uint64_t strides[1] = {(uint64_t)lv.kv.row_stride * 2};
      const uint32_t box[2] = {64u, 1u};
      if (encode_tmap(&tc[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lv.kv.base, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int max_cluster = max_cluster_for(reinterpret_cast<const void*>(kern), C::THREADS, C::SMEM_BYTES,
                                          which == 0 ? kClusterSlotMla0 : kClusterSlotMla1);
  if (max_cluster == 0) return cudaErrorUnknown;
  const int units = a.T * a.n_layers;
  const int tiles_max = (std::min(a.k, a.max_n) + kRows - 1) / kRows;
  int c = 1;
  while (c * 2 <= std::min(max_cluster, kMaxSplit) && c * 2 <= tiles_max &&
         (int64_t)units * c * 2 <= a.num_sms)
    c *= 2;
  // every block owns a value slice of >= 32 dims (one warp's lanes write one owner's slab)
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
  p.plan_early = a.plan_early ? 1 : 0;

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
  cfg.numAttrs = a.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, tq[0], tq[1], tq[2], tq[3], tc[0], tc[1], tc[2], tc[3], p);
}

}  // namespace

cudaError_t launch_sparse_mla(const MlaLaunch& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  // P^T lives in the last column block of a stage: the value dims end before it
  if (a.d_qk == 576 && a.d_v == 512) return launch_t<9, 4>(a, stream, 0);
  if (a.d_qk == 80 && a.d_v == 64) return launch_t<2, 1>(a, stream, 1);
  return cudaErrorInvalidValue;
}

}  // namespace dsa

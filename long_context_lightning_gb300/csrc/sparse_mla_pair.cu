// sparse_mla_pair.cu -- sparse MLA in MQA mode over the selected latent rows,
// for the 576-dim latent (512 value dims + 64 rope dims), with the columns of
// every selected row split over a pair of thread blocks.
//
// For query t and head h, over the selected positions s:
//   z_s = scale * Q[t, h, :576] . C[s, :576],  p = softmax(z),
//   O[t, h, :] = sum_s p_s C[s, :512],  LSE[t, h] = log sum_s exp(z_s)
// ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works /
// Model, sparse-MLA bullet: sparse MLA in MQA mode over the top-k tokens, all
// heads sharing the one latent row of a token; qk-nope 192 + rope 64 dims).
//
// Why a pair.  One block holding the whole 64-head query (72 KB) has room for
// a single 128-row tile (144 KB), so a tile's gather cannot overlap the
// previous tile's products.  Here block `half` of a pair holds the value dims
// [256 half, 256 half + 256) and rope dims [512 + 32 half, +32) of each row and
// the same columns of the query (36 KB), so two 72 KB stages fit.  Per tile:
//   S^T partial over this block's columns, M = 128 keys, N = 64 heads (18 MMAs)
//   exchange: the partial's columns of the peer's 32 heads go to the peer;
//             the peer's partial of this block's 32 heads comes back (DSMEM)
//   softmax:  this block owns 32 heads (reference m, running sum l)
//   P^T:      this block's 32 head columns are written here and in the peer,
//             with any reference move (scale factors) of this tile
//   O^T       += C^T . P^T over this block's 256 value dims (16 MMAs), so each
//             block accumulates its value half of all 64 heads.
// Both blocks add the same two fp32 partials, so the logits of a head are the
// same bits whichever block owns it.
//
// Softmax.  Probabilities are taken against a per-head reference that only
// moves when a score passes it by more than 2^16 (the first tile always moves
// it); the owner sends the move's factors with its P^T half, and each block
// rescales its own O^T columns of the moved heads before the PV.
//
// Row gather.  Rows land by 16-byte cp.async (a warp instruction moves four
// 128-byte row pieces; tile::gather4 issues at about 31 ns per instruction per
// warp, too slow for a 72 KB stage per tile): the four value blocks as [128
// rows x 64 dims] 128-byte-swizzled blocks, the rope half as [128 rows x 32
// dims] 64-byte-swizzled.  A stage is released in two parts as the two PV runs
// that read it complete (value blocks 0-1; value blocks 2-3 and the rope
// half).  Rows of later tiles are bulk-prefetched into L2 a few tiles ahead,
// half of them by each block, so the copies read L2.
//
// Split over pairs: the selected rows of a query are divided among the pairs
// of a cluster (1, 2, 4 or 8 pairs); the blocks that hold the same value half
// combine their partials through one exchange of bf16 slabs in distributed
// shared memory.
//
// Warp roles (416 threads, one block per SM):
//   warps 0..3   row gather: warp w owns value block w of each tile, warps 2
//                and 3 also half the rope half each, warp 0 the tile's valid
//                flags; L2 prefetch
//   warp 4       TMEM owner, query TMA, MMA issuer (one thread)
//   warps 5..12  S^T exchange, softmax of this block's 32 heads (one key and
//                16 heads per thread), P^T, O^T rescale; then the output
#include <algorithm>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 16.0f;  // move the reference only past 2^16
constexpr int kRows = 128;             // selected rows per tile
constexpr int kVBlk = kRows * 128;     // [128 rows x 64 dims] bf16
constexpr int kRBlk = kRows * 64;      // [128 rows x 32 dims] bf16
constexpr int kQBlk = 64 * 128;        // [64 heads x 64 dims] bf16
constexpr int kThreads = 416;
constexpr int kMaxPairs = 8;
constexpr int kPrefetchTiles = 6;      // tiles of rows prefetched into L2 ahead of their gather
constexpr int kSlabHeader = 512;       // (m, l) x 64 heads, fp32
constexpr int kXBytes = kRows * 32 * 4;       // the peer's partial of this block's heads
constexpr int kPBytes = kRows * 64 + 33 * 4;  // the peer's P^T half, its flag and factors
constexpr int kMLBytes = 64 * 4;              // the peer's (m, l) of its heads

// shared memory map (offsets from a 1024-aligned base)
constexpr int OFF_QV = 0;                               // 4 x [64 heads x 64 dims], 128-byte swizzle
constexpr int OFF_QR = OFF_QV + 4 * kQBlk;              // [64 heads x 32 dims], 64-byte swizzle
constexpr int OFF_ST = OFF_QR + 64 * 64;                // two stages
constexpr int STAGE = 4 * kVBlk + kRBlk;                // value blocks 0..3, then the rope half
constexpr int OFF_SRECV = OFF_ST + 2 * STAGE;           // [128 keys x 32 heads] fp32 from the peer
constexpr int OFF_PT = OFF_SRECV + kRows * 128;         // P^T [128 keys x 64 heads] bf16, 128-byte swizzle
constexpr int OFF_VALID = OFF_PT + kRows * 128;         // [2 stages][128] int
constexpr int OFF_MREF = OFF_VALID + 2 * kRows * 4;     // [32] reference of each own head (log2 units)
constexpr int OFF_ALPHA = OFF_MREF + 32 * 4;            // [32]
constexpr int OFF_RED = OFF_ALPHA + 32 * 4;             // [4 quadrants][32]
constexpr int MSG_WORDS = 36;                           // flag, 3 spare, 32 factors
constexpr int OFF_MSG = OFF_RED + 4 * 32 * 4;           // [2 tiles][own, peer][MSG_WORDS]
constexpr int OFF_ML = OFF_MSG + 2 * 2 * MSG_WORDS * 4; // m[64], l[64] of this pair
constexpr int OFF_INVL = OFF_ML + 128 * 4;              // 1/l [64]
constexpr int OFF_F = OFF_INVL + 64 * 4;                // combine weights [kMaxPairs][64]
constexpr int OFF_BAR = OFF_F + kMaxPairs * 64 * 4;
constexpr int N_BARS = 26;
constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;          // TMEM base, abort flag
constexpr int OFF_LAYER = OFF_MISC + 16;                // output, LSE, heads of this block's layer
constexpr int SMEM_BYTES = OFF_LAYER + 32 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(OFF_ST % 1024 == 0 && STAGE % 1024 == 0 && OFF_SRECV % 1024 == 0 && OFF_PT % 1024 == 0,
              "swizzled operands need 1024-byte alignment");
constexpr int TMEM_COLS = 256;  // O^T (two M-blocks x 64 heads) in [0, 128), S^T buffers at 128 and 192
constexpr int S_COL = 128;

// barrier indices
enum {
  B_FA = 0,         // [2] stage part a (value blocks 0-1) landed: 2 warp arrivals
  B_FB = 2,         // [2] stage part b (value blocks 2-3, rope half) landed: 2 warp arrivals
  B_V01FREE = 6,    // [2] value blocks 0-1 read by the PV (commit)
  B_V23FREE = 8,    // [2] value blocks 2-3 read by the PV, rope half by S^T (commit)
  B_SFULL = 10,     // [2] S^T partial formed (commit)
  B_SFREE = 12,     // [2] S^T buffer read by the softmax warps (8 arrivals)
  B_VALID = 14,     // [2] valid flags of the stage written (32 arrivals)
  B_XFULL = 16,     // the peer's partial of this block's heads landed (armed arrival + st.async bytes)
  B_PFULL = 18,     // both P^T halves and the peer's message written (8 local arrivals + st.async bytes)
  B_PVDONE = 19,    // both blocks' PV of the tile completed (2 multicast commits)
  B_RESC = 20,      // O^T columns rescaled (8 arrivals)
  B_Q = 21,         // query landed
  B_ML = 22,        // the peer's (m, l) landed (armed arrival + st.async bytes)
  B_READY = 23,     // same-half blocks of other pairs past their loops (remote arrivals)
  B_RECV = 24,      // slabs of the other pairs landed (bytes)
  B_DRAIN = 25,     // every issued MMA completed
};

struct LayerOut {
  __nv_bfloat16* out;
  float* lse;
  int32_t H;
  int32_t pad;
};

struct PairMaps {
  CUtensorMap qv[DSA_MAX_LAYERS];  // query value dims: box {64 dims, 64 heads, 1 query}, 128-byte swizzle
  CUtensorMap qr[DSA_MAX_LAYERS];  // query rope dims: box {32, 64, 1}, 64-byte swizzle
};

struct PairParams {
  MlaLayerView layer[DSA_MAX_LAYERS];
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

// Reduction of 16 values per lane across the warp by halving exchanges: lanes
// 2i and 2i+1 end with the reduction over all 32 lanes of element i.
template <bool MAX>
__device__ __forceinline__ float transpose_reduce16(const float (&x)[16], int lane) {
  float y[8];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float keep = hi ? x[8 + i] : x[i];
      const float send = hi ? x[i] : x[8 + i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      y[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int w = 8, n = 4; w >= 2; w >>= 1, n >>= 1) {
    const bool hi = lane & w;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float keep = hi ? y[n + i] : y[i];
      const float send = hi ? y[i] : y[n + i];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      y[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  const float got = __shfl_xor_sync(0xffffffffu, y[0], 1);
  return MAX ? fmaxf(y[0], got) : y[0] + got;
}

// Bounded wait with cluster-scope acquire that ignores the abort flag (the
// combine runs after every loop has ended).
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

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_pair_kernel(const __grid_constant__ PairMaps maps, const __grid_constant__ PairParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  int* valid_s = reinterpret_cast<int*>(smem + OFF_VALID);
  float* mref_s = reinterpret_cast<float*>(smem + OFF_MREF);
  float* alpha_s = reinterpret_cast<float*>(smem + OFF_ALPHA);
  float* red_s = reinterpret_cast<float*>(smem + OFF_RED);
  float* msg_s = reinterpret_cast<float*>(smem + OFF_MSG);
  float* ml_s = reinterpret_cast<float*>(smem + OFF_ML);
  float* invl_s = reinterpret_cast<float*>(smem + OFF_INVL);
  float* f_s = reinterpret_cast<float*>(smem + OFF_F);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const int half = (int)(crank & 1u);
  const int pair = (int)(crank >> 1);
  const int npairs = (int)(csize >> 1);
  const uint32_t peer = crank ^ 1u;
  const int t = blockIdx.y % p.T;
  const int li = blockIdx.y / p.T;
  const MlaLayerView& L = p.layer[li];
  const CUtensorMap* tm_qv = &maps.qv[li];
  const CUtensorMap* tm_qr = &maps.qr[li];
  // combine: the blocks of one value half split its 256 dims, `slice` each
  const int slice = 256 / npairs;
  const int ls = __ffs(slice) - 1;
  const uint32_t slab_bytes = (uint32_t)(kSlabHeader + slice * 32 * 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_FA + s), 2);
      mbar_init(bar(B_FB + s), 2);
      mbar_init(bar(B_V01FREE + s), 1);
      mbar_init(bar(B_V23FREE + s), 1);
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SFREE + s), 8);
      mbar_init(bar(B_VALID + s), 32);
    }
    mbar_init(bar(B_XFULL), 1);
    mbar_init(bar(B_PFULL), 8);
    mbar_init(bar(B_PVDONE), 2);
    mbar_init(bar(B_RESC), 8);
    mbar_init(bar(B_Q), 1);
    mbar_init(bar(B_ML), 1);
    mbar_init(bar(B_READY), npairs > 1 ? npairs - 1 : 1);
    mbar_init(bar(B_RECV), 1);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    LayerOut* lo = reinterpret_cast<LayerOut*>(smem + OFF_LAYER);
    lo->out = L.out;
    lo->lse = L.lse;
    lo->H = L.H;
    fence_mbar_init();
    // the peer's first partial and its (m, l) are counted in bytes; these
    // arrivals open the phases (later partials are armed as each one is read)
    mbar_arrive_expect_tx(bar(B_XFULL), kXBytes);
    mbar_arrive_expect_tx(bar(B_ML), kMLBytes);
    // the other pairs' slabs are counted in bytes; this arrival opens the phase
    if (npairs > 1) mbar_arrive_expect_tx(bar(B_RECV), (uint32_t)(npairs - 1) * slab_bytes);
  }
  if (threadIdx.x >= 160 && threadIdx.x < 192) mref_s[threadIdx.x - 160] = -INFINITY;
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // remote arrivals and stores may target this block from here on
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the query is a caller input: its load may overlap the previous grid
  if (warp == 4 && lane == 0) {
    mbar_arrive_expect_tx(bar(B_Q), 4 * kQBlk + 64 * 64);
    for (int kb = 0; kb < 4; ++kb)
      tma_load_3d(sbase + OFF_QV + kb * kQBlk, tm_qv, bar(B_Q), 256 * half + 64 * kb, 0, t);
    tma_load_3d(sbase + OFF_QR, tm_qr, bar(B_Q), 512 + 32 * half, 0, t);
  }

  // The plan is read before the wait when it was written two or more grids
  // back (complete before this grid could start); L2 loads, no stale L1.
  int n_t = 0, b = 0;
  int64_t seq_base = 0;
  auto read_plan = [&]() {
    n_t = __ldcg(p.q_n + t);
    b = __ldcg(p.q_seq + t);
    if (!L.kv.paged && b >= 0) seq_base = __ldg(L.kv.seq_start + b);
  };
  if (p.plan_early) read_plan();
  pdl_wait();  // positions and plan of the previous grids are complete from here on
  pdl_trigger();
  if (!p.plan_early) read_plan();
  const int nvalid = min(n_t, p.k);
  const int tiles = (nvalid + kRows - 1) / kRows;
  const int j0 = (int)((int64_t)tiles * pair / npairs);
  const int my_tiles = (int)((int64_t)tiles * (pair + 1) / npairs) - j0;

  if (warp < 4) {
    // ------------------------------------------------------------ row gather
    // Lane l of a gathering warp resolves rows l, l+32, l+64, l+96 of a tile
    // to pool rows (r4[k] = row 32k + l).
    const int32_t* idx_row = p.idx + (int64_t)t * p.ld_idx;
    int32_t r4[4];
    bool v4[4];
    auto resolve = [&](int jj) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = (j0 + jj) * kRows + 32 * k + lane;
        int pos = e < nvalid ? __ldg(idx_row + e) : -1;
        if (pos >= n_t || pos < -1) {
          if (warp == 0) atomicOr(p.err, DEV_ERR_BAD_INDEX);
          pos = -1;
        }
        int64_t row = -1;
        if (pos >= 0) {
          if (L.kv.paged) {
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
    const char* pool = reinterpret_cast<const char*>(L.kv.base);
    const int64_t pitch = L.kv.row_stride * 2;  // bytes between pool rows
    bool bad = false;
    auto issue = [&](int jj) {
      const int s = jj & 1;
      const uint32_t par = ((uint32_t)(jj >> 1) & 1u) ^ 1u;  // phase of this stage's previous use
      const uint32_t st_base = sbase + OFF_ST + s * STAGE;
      const int kb = warp;
      if (jj >= 2) bad |= !mbar_wait(bar((kb < 2 ? B_V01FREE : B_V23FREE) + s), par, abort_flag, p.err);
      if (warp == 0) {
        // the previous tile of this stage has finished its PV: its softmax read these
#pragma unroll
        for (int k = 0; k < 4; ++k) valid_s[s * kRows + 32 * k + lane] = v4[k];
        mbar_arrive(bar(B_VALID + s));
      }
      if (!bad) {
        // value block kb: instruction i moves rows 4i..4i+3, eight lanes (16-byte
        // chunks c) per row
        const int c = lane & 7;
        const char* src0 = pool + (256 * half + 64 * kb) * 2 + c * 16;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int row = 4 * i + (lane >> 3);
          const int32_t pr = __shfl_sync(0xffffffffu, r4[i >> 3], row & 31);  // i >> 3 is a constant here
          cp_async_16(st_base + kb * kVBlk + row * 128 + ((c ^ (row & 7)) << 4), src0 + (int64_t)pr * pitch, 16);
        }
        if (warp >= 2) {
          // rope half, rows 64 (w - 2) .. +63: instruction i moves eight rows, four
          // lanes (16-byte chunks c) per row
          const int cr = lane & 3;
          const char* srcr = pool + (512 + 32 * half) * 2 + cr * 16;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int row = 64 * (warp - 2) + 8 * i + (lane >> 2);
            const int32_t src_k = warp == 2 ? (i < 4 ? r4[0] : r4[1]) : (i < 4 ? r4[2] : r4[3]);  // r4[row >> 5]
            const int32_t pr = __shfl_sync(0xffffffffu, src_k, row & 31);
            cp_async_16(st_base + 4 * kVBlk + row * 64 + ((cr ^ ((row >> 1) & 3)) << 4), srcr + (int64_t)pr * pitch,
                        16);
          }
        }
      }
      cp_async_commit();
      cp_async_wait_all();
      fence_proxy_async_smem();  // the tensor cores read what cp.async wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(bar((kb < 2 ? B_FA : B_FB) + s));
    };
    // rows of a later tile into L2: row 32k + l of the tile for k = warp, the
    // lanes of this block's parity, so that the pair prefetches each row once
    auto prefetch = [&](int jj) {
      resolve(jj);
      int32_t rp = r4[0];
      bool vp = v4[0];
#pragma unroll
      for (int k = 1; k < 4; ++k)
        if (warp == k) {
          rp = r4[k];
          vp = v4[k];
        }
      if (vp && (lane & 1) == half && !bad) prefetch_l2_bulk(L.kv.base + (int64_t)rp * L.kv.row_stride, 576u * 2u);
    };
    const int first = min(my_tiles, 2);
    for (int jj = 0; jj < first; ++jj) {
      resolve(jj);
      issue(jj);
    }
    for (int jj = 2; jj < min(my_tiles, 2 + kPrefetchTiles); ++jj) prefetch(jj);
    for (int jj = 2; jj < my_tiles; ++jj) {
      resolve(jj);
      issue(jj);
      if (jj + kPrefetchTiles < my_tiles) prefetch(jj + kPrefetchTiles);
    }
  } else if (warp == 4) {
    // ---------------------------------------------- query TMA + MMA issuer
    if (lane == 0) {
      bool bad = !mbar_wait(bar(B_Q), 0, abort_flag, p.err);
      if (bad) mbar_wait_drain(bar(B_Q), 0);  // the query copy lands before the block may exit
      constexpr uint32_t idesc_s = mma_idesc_bf16(128, 64, false, false);
      constexpr uint32_t idesc_o = mma_idesc_bf16(128, 64, true, true);
      const uint64_t dqv = smem_desc_sw128(sbase + OFF_QV, 16, 1024);
      const uint64_t dqr = smem_desc_sw64(sbase + OFF_QR, 512);
      const uint64_t dp = smem_desc_sw128(sbase + OFF_PT, 16, 1024);  // P^T, MN-major, N = 64 in one block
      const uint16_t pair_mask = (uint16_t)(3u << (2 * pair));
      int ns = 0, npv = 0, nresc = 0, part = 0;
      uint64_t t_last = globaltimer_ns();
      uint32_t spin = 0;
      // Issue, in readiness order, the S^T runs (part a, part b) and the PV
      // runs; each run is one unbroken sequence of MMAs.  A PV is preferred:
      // it releases stage memory for the gather.
      while (npv < my_tiles && !bad) {
        bool did = false;
        if (npv < ns && mbar_test_wait_cluster(bar(B_PFULL), (uint32_t)npv & 1u)) {
          fence_proxy_async_smem();  // the peer's P^T half came by st.async
          tc_fence_after();
          const int* msg = reinterpret_cast<const int*>(msg_s + (npv & 1) * 2 * MSG_WORDS);
          if ((msg[0] | msg[MSG_WORDS]) != 0) {  // a reference moved: O^T is rescaled first
            if (!mbar_wait(bar(B_RESC), (uint32_t)nresc & 1u, abort_flag, p.err)) {
              bad = true;
              break;
            }
            ++nresc;
            tc_fence_after();
          }
          const int s = npv & 1;
          const uint64_t dv = smem_desc_sw128(sbase + OFF_ST + s * STAGE, kVBlk, 1024);  // C^T, MN-major
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16(tmem + 64 * mb, dv + (uint64_t)((2 * mb * kVBlk + kk * 2048) >> 4),
                       dp + (uint64_t)((kk * 2048) >> 4), idesc_o, (npv | kk) != 0);
            mma_commit(bar((mb == 0 ? B_V01FREE : B_V23FREE) + s));
          }
          mma_commit_mc(bar(B_PVDONE), pair_mask);  // this block's PV done, told to both blocks
          ++npv;
          did = true;
        } else if (ns < my_tiles) {
          const int s = ns & 1;
          const uint32_t ph = (uint32_t)(ns >> 1) & 1u;
          const uint32_t vb = sbase + OFF_ST + s * STAGE;
          const uint32_t scol = tmem + S_COL + 64 * (ns & 1);
          const uint64_t dk = smem_desc_sw128(vb, 16, 1024);
          if (part == 0) {
            if (mbar_test_wait(bar(B_FA + s), ph) &&
                (ns < 2 || mbar_test_wait(bar(B_SFREE + (ns & 1)), ph ^ 1u))) {
              tc_fence_after();
#pragma unroll
              for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_bf16(scol, dk + (uint64_t)((kb * kVBlk + kk * 32) >> 4),
                           dqv + (uint64_t)((kb * kQBlk + kk * 32) >> 4), idesc_s, (kb | kk) != 0);
              part = 1;
              did = true;
            }
          } else if (mbar_test_wait(bar(B_FB + s), ph)) {
            tc_fence_after();
#pragma unroll
            for (int kb = 2; kb < 4; ++kb)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16(scol, dk + (uint64_t)((kb * kVBlk + kk * 32) >> 4),
                         dqv + (uint64_t)((kb * kQBlk + kk * 32) >> 4), idesc_s, 1u);
            const uint64_t dr = smem_desc_sw64(vb + 4 * kVBlk, 512);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
              mma_bf16(scol, dr + (uint64_t)((kk * 32) >> 4), dqr + (uint64_t)((kk * 32) >> 4), idesc_s, 1u);
            mma_commit(bar(B_SFULL + (ns & 1)));
            part = 0;
            ++ns;
            did = true;
          }
        }
        if (did) {
          t_last = globaltimer_ns();
          spin = 0;
        } else if ((++spin & 63u) == 0) {
          if (*abort_flag) {
            bad = true;
          } else if (globaltimer_ns() - t_last > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(p.err, DEV_ERR_TIMEOUT);
            bad = true;
          }
        }
      }
      mma_commit(bar(B_DRAIN));
      mbar_wait_drain(bar(B_DRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int quad = warp & 3;           // TMEM lanes 32*quad .. +31 (keys of the tile)
    const int g = (warp - 5) >> 2;       // this thread's 16 of the block's 32 heads
    const int st = threadIdx.x - 160;    // 0..255
    const int srow = quad * 32 + lane;   // key of the tile held by this lane
    const int own0 = 32 * half + 16 * g;         // own heads (absolute index)
    const int oth0 = 32 * (half ^ 1) + 16 * g;   // the peer's matching heads
    const float c = L.scale * kLog2e;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t srecv_row = sbase + OFF_SRECV + srow * 128;
    const uint32_t pt_row = sbase + OFF_PT + srow * 128;
    float lsum[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) lsum[i] = 0.f;
    bool bad = false;
    for (int jj = 0; jj < my_tiles; ++jj) {
      const int bs = jj & 1;
      const uint32_t ph = (uint32_t)(jj >> 1) & 1u;
      bad |= !mbar_wait(bar(B_SFULL + bs), ph, abort_flag, p.err);
      tc_fence_after();
      const uint32_t scol = lane_base + S_COL + 64 * bs;
      uint32_t r[16];
      // the peer's heads of this block's partial go to the peer.  Its buffer is
      // free: the peer read the previous partial before it sent its P^T half of
      // the previous tile, which this thread waited for (st.async completes
      // with release semantics)
      tmem_ld16(scol + oth0, r);
      tmem_wait_ld();
      if (!bad) {
        const uint32_t xbar = dsmem_addr(bar(B_XFULL), peer);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t a = srecv_row + ((uint32_t)((4 * g + i) ^ (srow & 7)) << 4);
          st_async_v4(dsmem_addr(a, peer), r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3], xbar);
        }
      }
      // this block's heads: own partial plus the peer's partial
      tmem_ld16(scol + own0, r);
      tmem_wait_ld();
      bad |= !mbar_wait_cl(bar(B_XFULL), (uint32_t)jj & 1u, abort_flag, p.err);
      float x[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = ld_shared_v4(srecv_row + ((uint32_t)((4 * g + i) ^ (srow & 7)) << 4));
        x[4 * i] = __uint_as_float(r[4 * i]) + __uint_as_float(v.x);
        x[4 * i + 1] = __uint_as_float(r[4 * i + 1]) + __uint_as_float(v.y);
        x[4 * i + 2] = __uint_as_float(r[4 * i + 2]) + __uint_as_float(v.z);
        x[4 * i + 3] = __uint_as_float(r[4 * i + 3]) + __uint_as_float(v.w);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // every warp has passed this phase before the peer may send the next
        // partial (it waits for this tile's P^T half first), so the next phase
        // can be armed now
        if (warp == 5 && jj + 1 < my_tiles) mbar_arrive_expect_tx(bar(B_XFULL), kXBytes);
        mbar_arrive(bar(B_SFREE + bs));  // S^T buffer free for the tile after next
      }
      bad |= !mbar_wait(bar(B_VALID + bs), ph, abort_flag, p.err);
      const bool kv = valid_s[bs * kRows + srow] != 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = kv ? x[i] * c : -INFINITY;
      bool over = false;
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(mref_s + 16 * g + i);
        over |= (x[i] > m4.x + kRescaleLog2) | (x[i + 1] > m4.y + kRescaleLog2) | (x[i + 2] > m4.z + kRescaleLog2) |
                (x[i + 3] > m4.w + kRescaleLog2);
      }
      bool moved = false;
      if (bar_red_or(4, 256, over)) {
        // move the reference of every own head whose tile max passed it
        const float mx = transpose_reduce16<true>(x, lane);
        if ((lane & 1) == 0) red_s[quad * 32 + 16 * g + (lane >> 1)] = mx;
        named_bar_sync(3, 256);
        bool resc = false;
        if (st < 32) {
          const float mt = fmaxf(fmaxf(red_s[st], red_s[32 + st]), fmaxf(red_s[64 + st], red_s[96 + st]));
          const float mr = mref_s[st];
          float alpha = 1.f;
          if (mt > mr + kRescaleLog2 || (mr == -INFINITY && mt > -INFINITY)) {
            alpha = (mr == -INFINITY) ? 0.f : ex2_approx(mr - mt);
            mref_s[st] = mt;
            resc = mr != -INFINITY;
          }
          alpha_s[st] = alpha;
        }
        moved = bar_red_or(4, 256, resc);
#pragma unroll
        for (int i = 0; i < 16; ++i) lsum[i] *= alpha_s[16 * g + i];
      }
      // probabilities of this key for the own heads (bf16 pairs), running sums
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float2 m2 = *reinterpret_cast<const float2*>(mref_s + 16 * g + i);
        const float pa = x[i] == -INFINITY ? 0.f : ex2_approx(x[i] - m2.x);
        const float pb = x[i + 1] == -INFINITY ? 0.f : ex2_approx(x[i + 1] - m2.y);
        lsum[i] += pa;
        lsum[i + 1] += pb;
        w[i / 2] = pack_bf16x2(pa, pb);
      }
      // P^T here and in the peer is free once both blocks' PV of the previous tile completed
      if (jj >= 1) bad |= !mbar_wait_cl(bar(B_PVDONE), (uint32_t)(jj - 1) & 1u, abort_flag, p.err);
      float* msg_own = msg_s + bs * 2 * MSG_WORDS;
      const uint32_t msg_peer = dsmem_addr(smem_u32(msg_own + MSG_WORDS), peer);
      const uint32_t pbar = dsmem_addr(bar(B_PFULL), peer);
      if (st < 32) {
        const float a = moved ? alpha_s[st] : 1.f;
        msg_own[4 + st] = a;
        if (!bad) st_async_b32(msg_peer + (uint32_t)(4 + st) * 4u, __float_as_uint(a), pbar);
      }
      if (st == 0) {
        reinterpret_cast<int*>(msg_own)[0] = moved ? 1 : 0;
        if (!bad) st_async_b32(msg_peer, moved ? 1u : 0u, pbar);
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint32_t a = pt_row + ((uint32_t)((4 * half + 2 * g + cc) ^ (srow & 7)) << 4);
        st_shared_v4(a, w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
        if (!bad) st_async_v4(dsmem_addr(a, peer), w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3], pbar);
      }
      fence_proxy_async_smem();  // this block's tensor core reads the P^T written here
      __syncwarp();
      if (lane == 0) {
        // the peer's half and message arrive as bytes on this phase
        if (warp == 5) mbar_arrive_expect_tx(bar(B_PFULL), kPBytes);
        else mbar_arrive(bar(B_PFULL));
      }
      // a reference moved in either block: rescale this block's O^T columns of
      // the moved heads before the PV (the previous PV has completed)
      bad |= !mbar_wait_cl(bar(B_PFULL), (uint32_t)jj & 1u, abort_flag, p.err);
      int fl = 0;
      if (lane == 0) fl = reinterpret_cast<const int*>(msg_own)[0] | reinterpret_cast<const int*>(msg_own)[MSG_WORDS];
      fl = __shfl_sync(0xffffffffu, fl, 0);
      if (fl) {
        tc_fence_after();
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {  // M-block g, 16 head columns at a time
          const uint32_t col = lane_base + 64 * g + 16 * q4;
          uint32_t rr[16];
          tmem_ld16(col, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int h = 16 * q4 + i;
            const float a = msg_own[((h >> 5) == half ? 0 : MSG_WORDS) + 4 + (h & 31)];
            rr[i] = __float_as_uint(__uint_as_float(rr[i]) * a);
          }
          tmem_st16(col, rr);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_RESC));
      }
    }
    // (m, l) of the own heads over this pair's keys, shared with the peer
    {
      const float y = transpose_reduce16<false>(lsum, lane);
      if ((lane & 1) == 0) red_s[quad * 32 + 16 * g + (lane >> 1)] = y;
    }
    named_bar_sync(3, 256);
    if (st < 32) {
      const int h = 32 * half + st;
      const float l = red_s[st] + red_s[32 + st] + red_s[64 + st] + red_s[96 + st];
      const float m = mref_s[st];
      ml_s[h] = m;
      ml_s[64 + h] = l;
      const uint32_t mlbar = dsmem_addr(bar(B_ML), peer);
      st_async_b32(dsmem_addr(smem_u32(ml_s + h), peer), __float_as_uint(m), mlbar);
      st_async_b32(dsmem_addr(smem_u32(ml_s + 64 + h), peer), __float_as_uint(l), mlbar);
    }
    bad |= !mbar_wait_cl(bar(B_ML), 0, abort_flag, p.err);
    if (my_tiles > 0) bad |= !mbar_wait_cl(bar(B_PVDONE), (uint32_t)(my_tiles - 1) & 1u, abort_flag, p.err);
    tc_fence_after();
  }

  // ----------------------------------------------------------- the output
  __syncthreads();  // every role is past its loop: the stages are free
  const LayerOut lo = *reinterpret_cast<const LayerOut*>(smem + OFF_LAYER);
  if (npairs == 1) {
    if (warp >= 5) {
      const int quad = warp & 3, g = (warp - 5) >> 2, st = threadIdx.x - 160;
      const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
      if (st < 64) {
        const float l = ml_s[64 + st];
        invl_s[st] = l > 0.f ? 1.f / l : 0.f;
        if (half == 0 && lo.lse != nullptr && st < lo.H)
          lo.lse[(int64_t)t * lo.H + st] = l > 0.f ? (ml_s[st] + lg2_approx(l)) * kLn2 : -INFINITY;
      }
      named_bar_sync(3, 256);
      const int v = 256 * half + 128 * g + 32 * quad + lane;  // TMEM lane = value dim of M-block g
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t r[16];
        if (my_tiles > 0) {
          tmem_ld16(lane_base + 64 * g + 16 * q4, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int h = 16 * q4 + i;
          if (h < lo.H)
            lo.out[((int64_t)t * lo.H + h) * 512 + v] = __float2bfloat16_rn(__uint_as_float(r[i]) * invl_s[h]);
        }
      }
    }
  } else {
    // ------------------------------------------- combine over the pairs
    // The blocks holding value half `half` (ranks 2o + half) split its 256
    // dims, `slice` each.  recv: [source pair][slab], send: [owner pair][slab];
    // a slab is the source's (m, l) of all 64 heads, then one row per head pair
    // of the owner's slice, each word the pair as two bf16.
    uint8_t* recv = smem + OFF_ST;
    uint8_t* send = recv + npairs * slab_bytes;
    if (threadIdx.x == 0)
      for (int o = 0; o < npairs; ++o)
        if (o != pair) mbar_arrive_remote(dsmem_addr(bar(B_READY), (uint32_t)(2 * o + half)));
    if (warp >= 5) {
      const int quad = warp & 3, g = (warp - 5) >> 2, st = threadIdx.x - 160;
      const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
      if (st < 64) {
        for (int o = 0; o < npairs; ++o) {
          float* hdr = reinterpret_cast<float*>(o == pair ? recv + pair * slab_bytes : send + o * slab_bytes);
          hdr[st] = ml_s[st];
          hdr[64 + st] = ml_s[64 + st];
        }
      }
      {
        const int vq = 128 * g + 32 * quad;  // this warp's first value dim within the half
        const int owner = vq >> ls;          // a slice holds whole warps (>= 32 dims)
        const int vv = vq - (owner << ls) + lane;
        uint8_t* slab = owner == pair ? recv + pair * slab_bytes : send + owner * slab_bytes;
        uint32_t* col = reinterpret_cast<uint32_t*>(slab + kSlabHeader) + vv;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t r[16];
          if (my_tiles > 0) {
            tmem_ld16(lane_base + 64 * g + 16 * q4, r);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            col[(8 * q4 + i) * slice] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        }
      }
      fence_proxy_async_smem();  // the slabs are read by the bulk-copy engine
      named_bar_sync(3, 256);
      if (st == 0) {
        // a peer's stages may be overwritten only after its own loop has ended
        if (mbar_wait_cluster(bar(B_READY), 0, p.err)) {
          for (int o = 0; o < npairs; ++o) {
            if (o == pair) continue;
            const uint32_t dst = (uint32_t)(2 * o + half);
            bulk_copy_smem_to_peer(dsmem_addr(smem_u32(recv + pair * slab_bytes), dst),
                                   smem_u32(send + o * slab_bytes), slab_bytes, dsmem_addr(bar(B_RECV), dst));
          }
        }
      }
      const bool ok = mbar_wait_cluster(bar(B_RECV), 0, p.err);  // every source's slab has landed
      // weight of each source per head: four threads per head, each with the
      // sources sub and sub + 4; max and sum over a head's sources by shuffles
      {
        const int h = st >> 2, sub = st & 3;
        const float* h0p = reinterpret_cast<const float*>(recv + sub * slab_bytes);
        const float* h1p = reinterpret_cast<const float*>(recv + (sub + 4) * slab_bytes);
        const bool has0 = sub < npairs, has1 = sub + 4 < npairs;
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
      named_bar_sync(3, 256);
      // this block's slice of every head: one head pair and four value dims per
      // item (one 16-byte load per source, one 8-byte store per head)
      const int v0 = 256 * half + pair * slice;
      const int lvg = ls - 2;
      const int items = 32 << lvg;
      const float2* fw = reinterpret_cast<const float2*>(f_s);  // [source][head pair]
      for (int it = st; it < items; it += 256) {
        const int hp = it >> lvg;
        const int vg = it & ((1 << lvg) - 1);
        const int h = 2 * hp;
        if (h >= lo.H) continue;
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < kMaxPairs; ++r) {
          if (r < npairs) {
            const uint4 wv = *reinterpret_cast<const uint4*>(recv + r * slab_bytes + kSlabHeader +
                                                              (size_t)(hp * slice + 4 * vg) * 4);
            const float2 f2 = fw[r * 32 + hp];
            const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              a0[j] = fmaf(f2.x, bf16lo_to_f32(ws[j]), a0[j]);
              a1[j] = fmaf(f2.y, bf16hi_to_f32(ws[j]), a1[j]);
            }
          }
        }
        __nv_bfloat16* o0 = lo.out + ((int64_t)t * lo.H + h) * 512 + v0 + 4 * vg;
        *reinterpret_cast<uint2*>(o0) = make_uint2(pack_bf16x2(a0[0], a0[1]), pack_bf16x2(a0[2], a0[3]));
        if (h + 1 < lo.H)
          *reinterpret_cast<uint2*>(o0 + 512) = make_uint2(pack_bf16x2(a1[0], a1[1]), pack_bf16x2(a1[2], a1[3]));
      }
    }
  }
  // no block may leave while a peer could still read or write its shared memory
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_sparse_mla_pair(const MlaLaunch& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  if (a.d_qk != 576 || a.d_v != 512) return cudaErrorInvalidValue;
  auto kern = sparse_mla_pair_kernel;
  PairMaps maps;
  for (int l = 0; l < DSA_MAX_LAYERS; ++l) {
    const MlaLayerView& lv = a.layer[l < a.n_layers ? l : 0];
    {
      const uint64_t dims[3] = {576u, (uint64_t)lv.H, (uint64_t)a.T};
      const uint64_t strides[2] = {576u * 2u, (uint64_t)576 * lv.H * 2};
      const uint32_t box_v[3] = {64u, 64u, 1u};
      const uint32_t box_r[3] = {32u, 64u, 1u};
      if (encode_tmap(&maps.qv[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, lv.q, dims, strides, box_v,
                      CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
          encode_tmap(&maps.qr[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, lv.q, dims, strides, box_r,
                      CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int max_cluster = max_cluster_for(reinterpret_cast<const void*>(kern), kThreads, SMEM_BYTES,
                                          kClusterSlotMla0);
  if (max_cluster == 0) return cudaErrorUnknown;
  // pairs per query (and layer): as many as the SMs hold with every unit's
  // cluster resident at once, at least one tile each
  const int units = a.T * a.n_layers;
  const int tiles_max = (std::min(a.k, a.max_n) + kRows - 1) / kRows;
  int np = 1;
  while (np * 2 <= std::min(max_cluster / 2, kMaxPairs) && np * 2 <= tiles_max &&
         (int64_t)units * np * 4 <= a.num_sms)
    np *= 2;

  PairParams p;
  for (int l = 0; l < DSA_MAX_LAYERS; ++l) p.layer[l] = a.layer[l < a.n_layers ? l : 0];
  p.idx = a.idx;
  p.ld_idx = a.ld_idx;
  p.k = a.k;
  p.T = a.T;
  p.q_seq = a.q_seq;
  p.q_n = a.q_n;
  p.err = a.err;
  p.plan_early = a.plan_early ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * np, units, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2 * np;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1] = pdl_attribute();
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

}  // namespace dsa

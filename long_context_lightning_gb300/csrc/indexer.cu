// indexer.cu -- lightning-indexer scores on tcgen05 tensor cores.
//
//   I[t, s] = sum_h w[t, h] * max(0, q_I[t, h, :] . k_I[s, :])
// ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works /
// Model, lightning-indexer bullet; "DeepSeek Sparse Attention", In the code:
// the indexer sums ReLU(q.k) with weights).
//
// One work item = 128 consecutive keys of one sequence x one group of G
// queries of that sequence.  The MMA puts the 128 keys on M (TMEM lanes) and
// the group's (query, head) pairs on N, so D[s, (q, h)] = q_I[q, h] . k_I[s]
// lands in TMEM with one key per lane: the epilogue thread that owns key s
// applies ReLU, the head weight and the sum over heads in registers, with no
// cross-thread reduction, and writes one fp32 score per (query, key).  The
// per-head logits never leave the SM.
//
// Warp roles (one block per SM, persistent over the work list):
//   warp 0      TMA producer: key tiles into a ring of stages, the group's
//               indexer queries into the B buffer
//   warp 1      TMEM owner and MMA issuer (one elected thread)
//   warps 2..   epilogue: four warps (one per TMEM lane quadrant) for
//               one-query groups, eight for four-query groups (two per
//               quadrant, each owning two of the queries, so the per-key
//               ReLU / weight / head-sum work of a tile is split two ways);
//               two accumulators in TMEM so the epilogue of item i overlaps
//               the MMA of item i+1
#include <algorithm>

#include "internal.cuh"

namespace dsa {
namespace {

template <int KB, int NH, int G>
struct IdxCfg {
  static constexpr int N = NH * G;                   // MMA N: (query, head) pairs
  static constexpr int A_BYTES = KB * 128 * 128;     // 128 keys x KB blocks of 64 dims
  static constexpr int B_BYTES = KB * N * 128;
  // two query buffers when they are small, so the next group's queries load
  // while the current group's last MMAs still read theirs
  static constexpr int BSLOTS = (G == 1) ? 2 : 1;
  static constexpr int SMEM_BUDGET = 220 * 1024;
  static constexpr int STAGES_FIT = (SMEM_BUDGET - BSLOTS * B_BYTES - 4096) / A_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int TMEM_COLS = (2 * N <= 32) ? 32 : (2 * N <= 64) ? 64 : (2 * N <= 128) ? 128 : (2 * N <= 256) ? 256 : 512;
  static constexpr int EPI_WARPS = (G > 1) ? 8 : 4;  // epilogue warps
  static constexpr int EPI = 32 * EPI_WARPS;
  static constexpr int QH = G * 4 / EPI_WARPS;         // queries per epilogue warp
  static constexpr int THREADS = 64 + EPI;
  // shared memory map (offsets from a 1024-aligned base)
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_W = OFF_B + BSLOTS * B_BYTES;        // fp32 [G][NH]
  static constexpr int OFF_BAR = OFF_W + G * NH * 4;
  static constexpr int N_BARS = 2 * STAGES + 2 * BSLOTS + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;         // tmem base, abort flag
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;       // + alignment slack
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "tcgen05 M=128 needs N in [16, 256], multiple of 16");
  static_assert(STAGES >= 2, "ring too shallow");
};

struct IdxParams {
  CacheView k;
  const float* w;
  int32_t H;
  int32_t T;
  float* scores;
  int64_t ld;
  PlanView plan;
  int* err;
  int32_t keys_once;  // key tiles are read once: they enter L2 as evict-first, so the
                      // scores written meanwhile stay there for the top-k
};

// Work item -> group: the last g with start[g] <= item (start is non-decreasing,
// start[0] = 0).  One warp narrows the range 32-fold per round of loads.
__device__ __forceinline__ int find_group_warp(const int32_t* start, int n_groups, int item) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = n_groups - 1;
  while (hi - lo > 31) {
    const int q = lo + (int)((int64_t)(hi - lo) * lane / 31);
    const unsigned m = __ballot_sync(0xffffffffu, __ldg(start + q) <= item);
    const int last = 31 - __clz(m);  // lane 0 probes lo, which always qualifies
    const int nlo = __shfl_sync(0xffffffffu, q, last);
    const int nhi = last < 31 ? __shfl_sync(0xffffffffu, q, min(last + 1, 31)) - 1 : hi;
    lo = nlo;
    hi = max(nhi, nlo);
  }
  const int q = lo + lane;
  const unsigned m = __ballot_sync(0xffffffffu, q <= hi && __ldg(start + q) <= item);
  return lo + (31 - __clz(m));
}

template <int KB, int NH, int G>
__global__ void __launch_bounds__(IdxCfg<KB, NH, G>::THREADS, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   IdxParams p) {
  using C = IdxCfg<KB, NH, G>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  float* w_s = reinterpret_cast<float*>(smem + C::OFF_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* first_group = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);

  auto bar_a_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_a_empty = [&](int s) { return smem_u32(bars + C::STAGES + s); };
  auto bar_b_full = [&](int u) { return smem_u32(bars + 2 * C::STAGES + u); };
  auto bar_b_empty = [&](int u) { return smem_u32(bars + 2 * C::STAGES + C::BSLOTS + u); };
  constexpr int kAccBar = 2 * C::STAGES + 2 * C::BSLOTS;
  auto bar_acc_full = [&](int a) { return smem_u32(bars + kAccBar + a); };
  auto bar_acc_empty = [&](int a) { return smem_u32(bars + kAccBar + 2 + a); };
  const uint32_t bar_drain = smem_u32(bars + kAccBar + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_a_full(s), 1);
      mbar_init(bar_a_empty(s), 1);
    }
    for (int u = 0; u < C::BSLOTS; ++u) {
      mbar_init(bar_b_full(u), 1);
      mbar_init(bar_b_empty(u), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_acc_full(a), 1);
      mbar_init(bar_acc_empty(a), C::EPI);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_q);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();     // the plan (previous grid) is complete and visible from here on
  pdl_trigger();

  // this block's contiguous range of work items and the group of its first one
  const int n_groups = p.plan.header[0];
  const int total = p.plan.header[1];
  const int64_t nb = gridDim.x;
  const int w0 = (int)((int64_t)total * blockIdx.x / nb);
  const int w1 = (int)((int64_t)total * (blockIdx.x + 1) / nb);
  const int32_t* gstart = p.plan.g_tile_start;
  if (warp == 0) {
    const int g = (w0 < w1) ? find_group_warp(gstart, n_groups, w0) : 0;
    if (lane == 0) first_group[0] = g;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int g_first = first_group[0];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && w0 < w1) {
      const uint64_t once = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      int g = g_first;
      int g_next = __ldg(gstart + g + 1);
      int b_loads = 0;
      int4 gi = p.plan.g_info[g];
      int pend[C::STAGES];  // parity of the last load issued into each stage, or -1
      for (int s = 0; s < C::STAGES; ++s) pend[s] = -1;
      bool b_pending = false;
      for (int item = w0; item < w1; ++item) {
        bool new_group = (item == w0);
        while (item >= g_next) {
          ++g;
          g_next = __ldg(gstart + g + 1);
          new_group = true;
        }
        if (new_group) {
          gi = p.plan.g_info[g];
          const int u = b_loads % C::BSLOTS, use = b_loads / C::BSLOTS;
          if (use > 0 && !mbar_wait(bar_b_empty(u), (use - 1) & 1, abort_flag, p.err)) break;
          mbar_arrive_expect_tx(bar_b_full(u), C::B_BYTES);
          for (int kb = 0; kb < KB; ++kb)
            tma_load_3d(sbase + C::OFF_B + u * C::B_BYTES + kb * C::N * 128, &tm_q, bar_b_full(u), kb * 64, 0, gi.y);
          ++b_loads;
          b_pending = true;
        }
        const int kt = item - __ldg(gstart + g);
        if (!mbar_wait(bar_a_empty(stage), phase ^ 1, abort_flag, p.err)) break;
        const uint32_t dst = sbase + C::OFF_A + stage * C::A_BYTES;
        const int b = gi.x;
        if (!p.k.paged) {
          const int64_t row0 = __ldg(p.k.seq_start + b) + (int64_t)kt * 128;
          mbar_arrive_expect_tx(bar_a_full(stage), C::A_BYTES);
          for (int kb = 0; kb < KB; ++kb) {
            if (p.keys_once)
              tma_load_2d_hint(dst + kb * 128 * 128, &tm_k, bar_a_full(stage), kb * 64, (int32_t)row0, once);
            else
              tma_load_2d(dst + kb * 128 * 128, &tm_k, bar_a_full(stage), kb * 64, (int32_t)row0);
          }
        } else {
          // two 64-token pages per tile; pages past the sequence are not read
          const int n_pages = (gi.w + p.k.page_size - 1) / p.k.page_size;
          int64_t phys[2];
          int valid = 0;
          for (int h = 0; h < 2; ++h) {
            const int page = kt * 2 + h;
            phys[h] = -1;
            if (page < n_pages) {
              const int64_t v = __ldg(p.k.page_table + (int64_t)b * p.k.pt_stride + page);
              if (v >= 0 && (v + 1) * 64 <= p.k.num_rows) { phys[h] = v; ++valid; }
              else atomicOr(p.err, DEV_ERR_BAD_INDEX);
            }
          }
          mbar_arrive_expect_tx(bar_a_full(stage), valid * KB * 64 * 128);
          for (int h = 0; h < 2; ++h) {
            if (phys[h] < 0) continue;
            for (int kb = 0; kb < KB; ++kb) {
              if (p.keys_once)
                tma_load_2d_hint(dst + kb * 128 * 128 + h * 64 * 128, &tm_k, bar_a_full(stage), kb * 64,
                                 (int32_t)(phys[h] * 64), once);
              else
                tma_load_2d(dst + kb * 128 * 128 + h * 64 * 128, &tm_k, bar_a_full(stage), kb * 64,
                            (int32_t)(phys[h] * 64));
            }
          }
        }
        pend[stage] = (int)phase;
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
      if (*abort_flag) {  // let every issued copy land before the block goes away
        for (int s = 0; s < C::STAGES; ++s)
          if (pend[s] >= 0) mbar_wait_drain(bar_a_full(s), (uint32_t)pend[s]);
        if (b_pending)
          for (int v = b_loads > C::BSLOTS ? b_loads - C::BSLOTS : 0; v < b_loads; ++v)
            mbar_wait_drain(bar_b_full(v % C::BSLOTS), (uint32_t)((v / C::BSLOTS) & 1));
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0 && w0 < w1) {
      constexpr uint32_t idesc = mma_idesc_bf16(128, C::N, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int g = g_first;
      int g_next = __ldg(gstart + g + 1);
      int b_uses = 0;
      for (int item = w0; item < w1; ++item) {
        bool new_group = (item == w0);
        while (item >= g_next) {
          ++g;
          g_next = __ldg(gstart + g + 1);
          new_group = true;
        }
        if (new_group) {
          if (!mbar_wait(bar_b_full(b_uses % C::BSLOTS), (b_uses / C::BSLOTS) & 1, abort_flag, p.err)) break;
          ++b_uses;
        }
        if (!mbar_wait(bar_a_full(stage), phase, abort_flag, p.err)) break;
        if (!mbar_wait(bar_acc_empty(acc), acc_phase ^ 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t a_base = sbase + C::OFF_A + stage * C::A_BYTES;
        const uint32_t b_base = sbase + C::OFF_B + ((b_uses - 1) % C::BSLOTS) * C::B_BYTES;
        const uint32_t d = tmem + acc * C::N;
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_base + kb * 128 * 128 + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b_base + kb * C::N * 128 + kk * 32, 16, 1024);
            mma_bf16(d, ad, bd, idesc, (kb | kk) != 0);
          }
        }
        mma_commit(bar_a_empty(stage));
        mma_commit(bar_acc_full(acc));
        if (item + 1 >= g_next || item + 1 == w1) mma_commit(bar_b_empty((b_uses - 1) % C::BSLOTS));
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // drain: every issued MMA completes before TMEM is released
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int quad = warp & 3;           // TMEM lanes 32*quad .. +31
    const int row = quad * 32 + lane;    // key within the tile
    const int et = threadIdx.x - 64;     // 0 .. EPI-1
    const int qh0 = ((warp - 2) >> 2) * C::QH;  // this warp's first query of the group
    int acc = 0;
    uint32_t acc_phase = 0;
    bool bad = (w0 >= w1);
    int g = g_first;
    int g_next = bad ? 0 : __ldg(gstart + g + 1);
    int4 gi = make_int4(0, 0, 0, 0);
    int qn[C::QH];
    for (int item = w0; item < w1; ++item) {
      bool new_group = (item == w0);
      while (item >= g_next) {
        ++g;
        g_next = __ldg(gstart + g + 1);
        new_group = true;
      }
      if (new_group) {
        gi = p.plan.g_info[g];
        named_bar_sync(1, C::EPI);  // previous group's readers of w_s are done
        for (int i = et; i < G * NH; i += C::EPI) {
          const int q = i / NH, h = i % NH;
          float v = 0.f;
          if (q < gi.z && h < p.H) v = __ldg(p.w + (int64_t)(gi.y + q) * p.H + h);
          w_s[i] = v;
        }
#pragma unroll
        for (int qq = 0; qq < C::QH; ++qq) qn[qq] = (qh0 + qq < gi.z) ? p.plan.q_n[gi.y + qh0 + qq] : 0;
        named_bar_sync(1, C::EPI);
      }
      const int kt = item - __ldg(gstart + g);
      if (!bad && !mbar_wait(bar_acc_full(acc), acc_phase, abort_flag, p.err)) bad = true;
      tc_fence_after();
      const int64_t s = (int64_t)kt * 128 + row;
      const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + acc * C::N;
#pragma unroll
      for (int qq = 0; qq < C::QH; ++qq) {
        const int q = qh0 + qq;
        uint32_t r[NH];  // all head columns of this query, one wait
#pragma unroll
        for (int hc = 0; hc < NH / 16; ++hc)
          tmem_ld16(tbase + q * NH + hc * 16, *reinterpret_cast<uint32_t(*)[16]>(r + hc * 16));
        tmem_wait_ld();
        float part[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains over the heads
#pragma unroll
        for (int j = 0; j < NH; ++j)
          part[j & 3] = fmaf(w_s[q * NH + j], fmaxf(__uint_as_float(r[j]), 0.f), part[j & 3]);
        const float score = (part[0] + part[1]) + (part[2] + part[3]);
        if (!bad && q < gi.z && s < qn[qq]) p.scores[(int64_t)(gi.y + q) * p.ld + s] = score;
      }
      tc_fence_before();
      mbar_arrive(bar_acc_empty(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int KB, int NH, int G>
cudaError_t launch_t(const IndexerLaunch& a, cudaStream_t stream) {
  using C = IdxCfg<KB, NH, G>;
  CUtensorMap tm_k, tm_q;
  {
    const uint64_t dims[2] = {(uint64_t)a.d, (uint64_t)a.k.num_rows};
    const uint64_t strides[1] = {(uint64_t)a.k.row_stride * 2};
    const uint32_t box[2] = {64u, a.k.paged ? 64u : 128u};
    if (encode_tmap(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k.base, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)a.d, (uint64_t)a.H, (uint64_t)a.T};
    const uint64_t strides[2] = {(uint64_t)a.d * 2, (uint64_t)a.d * a.H * 2};
    const uint32_t box[3] = {64u, (uint32_t)NH, (uint32_t)G};
    if (encode_tmap(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  IdxParams p;
  p.k = a.k;
  p.w = a.w;
  p.H = a.H;
  p.T = a.T;
  p.scores = a.scores;
  p.ld = a.ld;
  p.plan = a.plan;
  p.err = a.err;
  p.keys_once = a.keys_once ? 1 : 0;
  cudaError_t e = cudaFuncSetAttribute(indexer_kernel<KB, NH, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // Upper bound of work items: every query group scans at most ceil(max_n/128)
  // tiles.  The grid is one block per SM; blocks with an empty range exit.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_sms, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute at = pdl_attribute();
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, indexer_kernel<KB, NH, G>, tm_k, tm_q, p);
}

}  // namespace

cudaError_t launch_indexer(const IndexerLaunch& a, cudaStream_t stream) {
  const int KB = a.d <= 64 ? 1 : 2;
  const int NH = a.H <= 16 ? 16 : 64;
  if (KB == 1 && NH == 16) return a.group == 1 ? launch_t<1, 16, 1>(a, stream) : launch_t<1, 16, 4>(a, stream);
  if (KB == 1 && NH == 64) return a.group == 1 ? launch_t<1, 64, 1>(a, stream) : launch_t<1, 64, 4>(a, stream);
  if (KB == 2 && NH == 16) return a.group == 1 ? launch_t<2, 16, 1>(a, stream) : launch_t<2, 16, 4>(a, stream);
  return a.group == 1 ? launch_t<2, 64, 1>(a, stream) : launch_t<2, 64, 4>(a, stream);
}

}  // namespace dsa

// hisparse.cu -- HBM as a least-recently-used cache of latent rows over host
// memory, for the rows a top-k selection asks for.
//
// "How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works /
// HiSparse (SGLang): the rows chosen by top-k that are missing from HBM are
// loaded from host DRAM, cold rows are evicted, and the loads for layer N
// overlap the execution of layer N-1 (each call is asynchronous on its stream,
// so a caller fetches layer N on one stream while layer N-1's attention runs on
// another).  The cache is read-only: host memory holds every row, so evicting
// a row needs no write-back.
//
// State (one device buffer, carved below): the slot of every host row (or
// -1), the host row in every slot (or -1), the least-recently-used order of the
// slots, the step at which each slot was last used, per-row first-request
// stamps, this step's misses and their slots, and counters.
//
// One fetch = four launches after the per-call plan:
//   lookup   every selected entry: stamp its host row with (step, entry index)
//            so the first request of a row is known, and mark resident rows'
//            slots used in this step
//   plan     one block: the misses in first-request order; the LRU order
//            split into [not used this step] ++ [used this step] (stable); the
//            first misses-many slots of the first part are the victims; new
//            order = [rest of the first part] ++ [used] ++ [victims]; tables
//            updated, evicted rows dropped
//   copy     one warp per miss: the host row into its slot (16-byte loads of
//            pinned host memory)
//   resolve  every selected entry: the slot now holding its row
#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kEntryThreads = 256;
constexpr int kCopyWarps = 8;

enum { ST_STEP = 0, ST_REQUESTS = 1, ST_HITS = 2, ST_MISSES = 3, ST_EVICTED = 4, ST_OVERFLOW = 5 };

struct HsState {
  int32_t* slot_of_row;  // [host_rows]
  uint64_t* claim;       // [host_rows]
  int32_t* row_of_slot;  // [capacity]
  int32_t* lru;          // [capacity] slots, least recently used first
  int32_t* lru_next;     // [capacity]
  int32_t* used;         // [capacity] step of the slot's last use
  int32_t* miss_rows;    // [capacity]
  int32_t* miss_slots;   // [capacity]
  int32_t* stats;        // [8]
};

size_t state_bytes(int64_t capacity, int64_t host_rows) {
  return align_up(4 * (size_t)host_rows, 256) + align_up(8 * (size_t)host_rows, 256) +
         6 * align_up(4 * (size_t)capacity, 256) + 256;
}

HsState carve(void* base, int64_t capacity, int64_t host_rows) {
  char* p = static_cast<char*>(base);
  HsState s;
  s.slot_of_row = reinterpret_cast<int32_t*>(p);
  p += align_up(4 * (size_t)host_rows, 256);
  s.claim = reinterpret_cast<uint64_t*>(p);
  p += align_up(8 * (size_t)host_rows, 256);
  int32_t** arr[6] = {&s.row_of_slot, &s.lru, &s.lru_next, &s.used, &s.miss_rows, &s.miss_slots};
  for (int i = 0; i < 6; ++i) {
    *arr[i] = reinterpret_cast<int32_t*>(p);
    p += align_up(4 * (size_t)capacity, 256);
  }
  s.stats = reinterpret_cast<int32_t*>(p);
  return s;
}

struct HsParams {
  HsState s;
  int32_t capacity;
  int64_t host_rows;
  int32_t row_elems;
  __nv_bfloat16* slot_pool;
  int64_t slot_stride;
  CacheView host;  // the layer's latent cache in host memory (device-accessible pointer)
  const int32_t* idx;
  int64_t ld_idx;
  int32_t k;
  int32_t T;
  const int32_t* q_seq;
  const int32_t* q_n;
  int32_t* slots;
  int64_t ld_slots;
  int* err;
};

__device__ __forceinline__ uint64_t claim_key(uint32_t step, uint32_t flat) {
  // a later step wins; within a step, the lowest entry index wins
  return ((uint64_t)step << 32) | (uint64_t)(0xffffffffu - flat);
}

// Host row of selection entry f = t * k + j, or -1 for an empty entry (-1) or
// a bad one (flagged when `flag`).
__device__ __forceinline__ int64_t entry_row(const HsParams& p, int f, bool flag) {
  const int t = f / p.k, j = f - t * p.k;
  const int n_t = p.q_n[t];
  if (j >= min(n_t, p.k)) return -1;
  const int pos = p.idx[(int64_t)t * p.ld_idx + j];
  if (pos == -1) return -1;
  if (pos < -1 || pos >= n_t) {
    if (flag) atomicOr(p.err, DEV_ERR_BAD_INDEX);
    return -1;
  }
  const int64_t row = cache_row(p.host, p.q_seq[t], pos);
  if (row < 0 || row >= p.host_rows) {
    if (flag) atomicOr(p.err, DEV_ERR_BAD_INDEX);
    return -1;
  }
  return row;
}

__global__ void hs_reset_kernel(HsState s, int32_t capacity, int64_t host_rows) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < host_rows; i += stride) {
    s.slot_of_row[i] = -1;
    s.claim[i] = 0;
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < capacity; i += stride) {
    s.row_of_slot[i] = -1;
    s.lru[i] = (int32_t)i;
    s.used[i] = 0;  // steps start at 1
  }
  if (blockIdx.x == 0 && threadIdx.x < 8) s.stats[threadIdx.x] = 0;
}

__global__ void __launch_bounds__(kEntryThreads) hs_lookup_kernel(HsParams p) {
  pdl_wait();  // the plan and the previous fetch are complete from here on
  pdl_trigger();
  const int f = blockIdx.x * kEntryThreads + threadIdx.x;
  if (f >= p.T * p.k) return;
  const uint32_t step = (uint32_t)p.s.stats[ST_STEP] + 1u;
  const int64_t row = entry_row(p, f, true);
  if (row < 0) return;
  atomicMax(reinterpret_cast<unsigned long long*>(p.s.claim + row), (unsigned long long)claim_key(step, (uint32_t)f));
  const int slot = p.s.slot_of_row[row];
  if (slot >= 0) p.s.used[slot] = (int32_t)step;
}

// Exclusive block-wide scan of one int per thread (all threads call it).
__device__ int scan_block(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int before = (warp ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kPlanThreads, 1) hs_plan_kernel(HsParams p) {
  __shared__ int warp_sums[32];
  __shared__ int s_overflow;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  const uint32_t step = (uint32_t)p.s.stats[ST_STEP] + 1u;
  const int cap = p.capacity;

  // (1) distinct requested rows in first-request order: misses compacted, hits counted
  int n_miss = 0, n_hit = 0;
  const int n_entries = p.T * p.k;
  for (int f0 = 0; f0 < n_entries; f0 += kPlanThreads) {
    const int f = f0 + tid;
    int miss = 0, hit = 0;
    int64_t row = -1;
    if (f < n_entries) {
      row = entry_row(p, f, false);
      if (row >= 0 && p.s.claim[row] == claim_key(step, (uint32_t)f)) {
        miss = p.s.slot_of_row[row] < 0;
        hit = !miss;
      }
    }
    int tot_m, tot_h;
    const int ex = scan_block(miss, warp_sums, &tot_m);
    scan_block(hit, warp_sums, &tot_h);
    if (miss && n_miss + ex < cap) p.s.miss_rows[n_miss + ex] = (int32_t)row;
    n_miss += tot_m;
    n_hit += tot_h;
  }
  // every requested row must fit: the slots used this step (n_hit) plus the misses
  if (tid == 0) s_overflow = (n_miss > cap - n_hit) ? 1 : 0;
  __syncthreads();
  if (s_overflow) {
    if (tid == 0) {
      atomicOr(p.err, DEV_ERR_CAPACITY);
      p.s.stats[ST_OVERFLOW] = 1;
      p.s.stats[ST_MISSES] = 0;
      p.s.stats[ST_STEP] = (int32_t)step;
    }
    return;
  }

  // (2) LRU order: [not used this step] ++ [used this step], both stable; the
  // first n_miss of the first part are the victims and go to the end
  int n_a = 0;
  for (int i0 = 0; i0 < cap; i0 += kPlanThreads) {
    const int i = i0 + tid;
    const int a = (i < cap && p.s.used[p.s.lru[i]] != (int32_t)step) ? 1 : 0;
    int tot;
    scan_block(a, warp_sums, &tot);
    n_a += tot;
  }
  int a_run = 0, b_run = 0, evicted = 0;
  for (int i0 = 0; i0 < cap; i0 += kPlanThreads) {
    const int i = i0 + tid;
    int slot = -1, is_a = 0, is_b = 0;
    if (i < cap) {
      slot = p.s.lru[i];
      is_a = p.s.used[slot] != (int32_t)step;
      is_b = !is_a;
    }
    int tot_a, tot_b, tot_e;
    const int ea = scan_block(is_a, warp_sums, &tot_a);
    const int eb = scan_block(is_b, warp_sums, &tot_b);
    int ev = 0;
    if (is_a) {
      const int a = a_run + ea;
      if (a < n_miss) {
        // victim a receives miss row a; its old row (if any) leaves HBM
        const int old = p.s.row_of_slot[slot];
        if (old >= 0) {
          p.s.slot_of_row[old] = -1;
          ev = 1;
        }
        const int row = p.s.miss_rows[a];
        p.s.row_of_slot[slot] = row;
        p.s.slot_of_row[row] = slot;
        p.s.used[slot] = (int32_t)step;
        p.s.miss_slots[a] = slot;
        p.s.lru_next[cap - n_miss + a] = slot;
      } else {
        p.s.lru_next[a - n_miss] = slot;
      }
    } else if (is_b) {
      p.s.lru_next[n_a - n_miss + b_run + eb] = slot;
    }
    scan_block(ev, warp_sums, &tot_e);
    a_run += tot_a;
    b_run += tot_b;
    evicted += tot_e;
  }
  __syncthreads();
  for (int i = tid; i < cap; i += kPlanThreads) p.s.lru[i] = p.s.lru_next[i];
  if (tid == 0) {
    p.s.stats[ST_REQUESTS] = n_hit + n_miss;
    p.s.stats[ST_HITS] = n_hit;
    p.s.stats[ST_MISSES] = n_miss;
    p.s.stats[ST_EVICTED] = evicted;
    p.s.stats[ST_OVERFLOW] = 0;
    p.s.stats[ST_STEP] = (int32_t)step;
  }
}

__global__ void __launch_bounds__(32 * kCopyWarps) hs_copy_kernel(HsParams p) {
  pdl_wait();
  pdl_trigger();
  const int a = blockIdx.x * kCopyWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (a >= p.s.stats[ST_MISSES]) return;
  const int64_t row = p.s.miss_rows[a];
  const int64_t slot = p.s.miss_slots[a];
  const uint4* src = reinterpret_cast<const uint4*>(p.host.base + row * p.host.row_stride);
  uint4* dst = reinterpret_cast<uint4*>(p.slot_pool + slot * p.slot_stride);
  for (int i = lane; i < p.row_elems / 8; i += 32) dst[i] = src[i];
}

__global__ void __launch_bounds__(kEntryThreads) hs_resolve_kernel(HsParams p) {
  pdl_wait();
  pdl_trigger();
  const int f = blockIdx.x * kEntryThreads + threadIdx.x;
  if (f >= p.T * p.k) return;
  const int t = f / p.k, j = f - t * p.k;
  const int64_t row = entry_row(p, f, false);
  p.slots[(int64_t)t * p.ld_slots + j] = row >= 0 ? p.s.slot_of_row[row] : -1;
}

__global__ void hs_resident_kernel(HsState s, int32_t capacity, int32_t* rows) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < capacity; i += gridDim.x * blockDim.x)
    rows[i] = s.row_of_slot[s.lru[i]];
}

cudaError_t launch_pdl(const void* kern, int grid, int block, void** args, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute at = pdl_attribute();
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace

size_t hisparse_state_bytes(int64_t capacity, int64_t host_rows) { return state_bytes(capacity, host_rows); }

cudaError_t launch_hisparse_reset(void* state, int32_t capacity, int64_t host_rows, cudaStream_t stream) {
  const HsState s = carve(state, capacity, host_rows);
  const int64_t n = std::max<int64_t>(host_rows, capacity);
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 4096);
  hs_reset_kernel<<<grid, 256, 0, stream>>>(s, capacity, host_rows);
  return cudaGetLastError();
}

cudaError_t launch_hisparse_fetch(const HisparseLaunch& a, cudaStream_t stream) {
  HsParams p;
  p.s = carve(a.state, a.capacity, a.host_rows);
  p.capacity = a.capacity;
  p.host_rows = a.host_rows;
  p.row_elems = a.row_elems;
  p.slot_pool = static_cast<__nv_bfloat16*>(a.slot_pool);
  p.slot_stride = a.slot_stride;
  p.host = a.host;
  p.idx = a.idx;
  p.ld_idx = a.ld_idx;
  p.k = a.k;
  p.T = a.T;
  p.q_seq = a.q_seq;
  p.q_n = a.q_n;
  p.slots = a.slots;
  p.ld_slots = a.ld_slots;
  p.err = a.err;
  void* args[] = {&p};
  const int n = a.T * a.k;
  const int entry_grid = (n + kEntryThreads - 1) / kEntryThreads;
  cudaError_t e;
  if ((e = launch_pdl(reinterpret_cast<const void*>(hs_lookup_kernel), entry_grid, kEntryThreads, args, stream)))
    return e;
  if ((e = launch_pdl(reinterpret_cast<const void*>(hs_plan_kernel), 1, kPlanThreads, args, stream))) return e;
  const int max_miss = std::min(n, a.capacity);
  if ((e = launch_pdl(reinterpret_cast<const void*>(hs_copy_kernel), std::max(1, (max_miss + kCopyWarps - 1) / kCopyWarps),
                      32 * kCopyWarps, args, stream)))
    return e;
  return launch_pdl(reinterpret_cast<const void*>(hs_resolve_kernel), entry_grid, kEntryThreads, args, stream);
}

cudaError_t launch_hisparse_resident(void* state, int32_t capacity, int64_t host_rows, int32_t* rows,
                                     cudaStream_t stream) {
  const HsState s = carve(state, capacity, host_rows);
  hs_resident_kernel<<<std::max(1, std::min((capacity + 255) / 256, 1024)), 256, 0, stream>>>(s, capacity, rows);
  return cudaGetLastError();
}

cudaError_t hisparse_read_stats(void* state, int32_t capacity, int64_t host_rows, int32_t* out8,
                                cudaStream_t stream) {
  const HsState s = carve(state, capacity, host_rows);
  cudaError_t e = cudaMemcpyAsync(out8, s.stats, 8 * sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace dsa

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
// One fetch = six launches after the per-call plan, each over many blocks
// except the scan:
//   lookup   every selected entry: stamp its host row with (step, entry index)
//            so the first request of a row is known, and mark resident rows'
//            slots used in this step
//   count    per chunk of 2048 entries: first-request misses and hits; per
//            chunk of 2048 LRU positions: slots not used in this step
//   scan     one block: chunk offsets, totals, the capacity check
//   scatter  misses to their place in first-request order; the LRU order
//            split into [not used this step] ++ [used this step] (stable); the
//            first misses-many slots of the first part are the victims (their
//            rows dropped); new order = [rest of the first part] ++ [used] ++
//            [victims], written to the other of two order buffers
//   copy     one warp per miss: bind the victim slot to the row and copy the
//            host row into it (16-byte loads of pinned host memory)
//   resolve  every selected entry: the slot now holding its row
#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kPer = 8;                     // items per thread in the count and scatter passes
constexpr int kChunk = kThreads * kPer;     // items per block there
constexpr int kScanThreads = 1024;
constexpr int kCopyWarps = 8;

enum {
  ST_STEP = 0, ST_REQUESTS = 1, ST_HITS = 2, ST_MISSES = 3, ST_EVICTED = 4, ST_OVERFLOW = 5,
  ST_PARITY = 6,   // which of the two order buffers is current
  ST_NOT_USED = 7  // slots not used in this step (this fetch's scan)
};

struct HsState {
  int32_t* slot_of_row;  // [host_rows]
  uint64_t* claim;       // [host_rows]
  int32_t* row_of_slot;  // [capacity]
  int32_t* lru[2];       // [capacity] each: slots, least recently used first; stats[ST_PARITY] picks the current
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
  int32_t** arr[6] = {&s.row_of_slot, &s.lru[0], &s.lru[1], &s.used, &s.miss_rows, &s.miss_slots};
  for (int i = 0; i < 6; ++i) {
    *arr[i] = reinterpret_cast<int32_t*>(p);
    p += align_up(4 * (size_t)capacity, 256);
  }
  s.stats = reinterpret_cast<int32_t*>(p);
  return s;
}

// Per-call chunk counts, carved from the caller's workspace after the plan.
struct Counts {
  int32_t* miss;  // [n_entry_chunks] misses per entry chunk, then (after the scan) their offsets
  int32_t* hit;   // [n_entry_chunks]
  int32_t* a;     // [n_lru_chunks] not-used slots per LRU chunk, then their offsets
};

int64_t entry_chunks(int64_t entries) { return (entries + kChunk - 1) / kChunk; }
int64_t lru_chunks(int64_t capacity) { return (capacity + kChunk - 1) / kChunk; }

size_t counts_bytes(int64_t entries, int64_t capacity) {
  return 2 * align_up(4 * (size_t)entry_chunks(entries), 256) + align_up(4 * (size_t)lru_chunks(capacity), 256);
}

Counts carve_counts(void* base, int64_t entries, int64_t capacity) {
  char* p = static_cast<char*>(base);
  Counts c;
  c.miss = reinterpret_cast<int32_t*>(p);
  p += align_up(4 * (size_t)entry_chunks(entries), 256);
  c.hit = reinterpret_cast<int32_t*>(p);
  p += align_up(4 * (size_t)entry_chunks(entries), 256);
  c.a = reinterpret_cast<int32_t*>(p);
  return c;
}

struct HsParams {
  HsState s;
  Counts c;
  int32_t n_entry_chunks;
  int32_t n_lru_chunks;
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

// Status of the kPer selection entries f0 .. f0 + kPer - 1 in this step:
// kind 1 = first request of a missing row, 2 = first request of a resident
// row, 0 = anything else (past the selection: kind 0, row -1).  Every load step is issued for all entries at once --
// context lengths, sequences and positions, then pool rows, then claims, then
// slots -- with indices clamped into range and the conditions applied after,
// so a thread waits four load latencies, not four per entry.
__device__ __forceinline__ void entry_kinds(const HsParams& p, int f0, uint32_t step, int64_t (&rows)[kPer],
                                            int (&kinds)[kPer]) {
  const int n_entries = p.T * p.k;
  int n_t[kPer], seq[kPer], pos[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int f = min(f0 + i, n_entries - 1);
    const int t = f / p.k, j = f - t * p.k;
    n_t[i] = __ldg(p.q_n + t);
    seq[i] = __ldg(p.q_seq + t);
    pos[i] = __ldg(p.idx + (int64_t)t * p.ld_idx + j);
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int f = f0 + i;
    const int j = f - (min(f, n_entries - 1) / p.k) * p.k;
    const bool ok = f < n_entries && j < min(n_t[i], p.k) && pos[i] >= 0 && pos[i] < n_t[i];
    const int64_t row = cache_row(p.host, seq[i], ok ? pos[i] : 0);
    rows[i] = (ok && row >= 0 && row < p.host_rows) ? row : -1;
  }
  uint64_t claim[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) claim[i] = rows[i] >= 0 ? p.s.claim[rows[i]] : 0ull;
  int slot[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const bool first = rows[i] >= 0 && claim[i] == claim_key(step, (uint32_t)(f0 + i));
    slot[i] = first ? p.s.slot_of_row[rows[i]] : 0;
    kinds[i] = first ? (slot[i] < 0 ? 1 : 2) : 0;
  }
}

// The kPer positions i0 .. i0 + kPer - 1 of an LRU order (two 16-byte loads;
// past the capacity: -2).
__device__ __forceinline__ void lru_slots(const int32_t* lru, int i0, int cap, int (&slots)[kPer]) {
  static_assert(kPer == 8, "two 16-byte loads per thread");
  if (i0 + kPer <= cap) {
    const int4 v0 = *reinterpret_cast<const int4*>(lru + i0);
    const int4 v1 = *reinterpret_cast<const int4*>(lru + i0 + 4);
    slots[0] = v0.x, slots[1] = v0.y, slots[2] = v0.z, slots[3] = v0.w;
    slots[4] = v1.x, slots[5] = v1.y, slots[6] = v1.z, slots[7] = v1.w;
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) slots[i] = i0 + i < cap ? lru[i0 + i] : -2;
  }
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

__global__ void hs_reset_kernel(HsState s, int32_t capacity, int64_t host_rows) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < host_rows; i += stride) {
    s.slot_of_row[i] = -1;
    s.claim[i] = 0;
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < capacity; i += stride) {
    s.row_of_slot[i] = -1;
    s.lru[0][i] = (int32_t)i;
    s.used[i] = 0;  // steps start at 1
  }
  if (blockIdx.x == 0 && threadIdx.x < 8) s.stats[threadIdx.x] = 0;
}

__global__ void __launch_bounds__(kThreads) hs_lookup_kernel(HsParams p) {
  pdl_wait();  // the plan and the previous fetch are complete from here on
  pdl_trigger();
  const int f = blockIdx.x * kThreads + threadIdx.x;
  if (f >= p.T * p.k) return;
  const uint32_t step = (uint32_t)p.s.stats[ST_STEP] + 1u;
  const int64_t row = entry_row(p, f, true);
  if (row < 0) return;
  atomicMax(reinterpret_cast<unsigned long long*>(p.s.claim + row), (unsigned long long)claim_key(step, (uint32_t)f));
  const int slot = p.s.slot_of_row[row];
  if (slot >= 0) p.s.used[slot] = (int32_t)step;
}

__global__ void __launch_bounds__(kThreads) hs_count_kernel(HsParams p) {
  __shared__ int warp_sums[32];
  pdl_wait();
  pdl_trigger();
  const uint32_t step = (uint32_t)p.s.stats[ST_STEP] + 1u;
  const int n_entries = p.T * p.k;
  if ((int)blockIdx.x < p.n_entry_chunks) {
    int miss = 0, hit = 0;
    const int f0 = blockIdx.x * kChunk + threadIdx.x * kPer;
    if (f0 < n_entries) {
      int64_t rows[kPer];
      int kinds[kPer];
      entry_kinds(p, f0, step, rows, kinds);
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        miss += kinds[i] == 1;
        hit += kinds[i] == 2;
      }
    }
    int tot_m, tot_h;
    scan_block(miss, warp_sums, &tot_m);
    scan_block(hit, warp_sums, &tot_h);
    if (threadIdx.x == 0) {
      p.c.miss[blockIdx.x] = tot_m;
      p.c.hit[blockIdx.x] = tot_h;
    }
  } else {
    const int chunk = blockIdx.x - p.n_entry_chunks;
    const int32_t* lru = p.s.lru[p.s.stats[ST_PARITY] & 1];
    int a = 0;
    const int i0 = chunk * kChunk + threadIdx.x * kPer;
    if (i0 < p.capacity) {
      int slots[kPer];
      lru_slots(lru, i0, p.capacity, slots);
      bool bad = false;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const bool in = (unsigned)slots[i] < (unsigned)p.capacity;
        bad |= !in && slots[i] != -2;  // the order is a permutation of the slots
        a += in && p.s.used[in ? slots[i] : 0] != (int32_t)step;
      }
      if (bad) atomicOr(p.err, DEV_ERR_BAD_INDEX);
    }
    int tot;
    scan_block(a, warp_sums, &tot);
    if (threadIdx.x == 0) p.c.a[chunk] = tot;
  }
}

// In-place exclusive scan of n ints by one block; returns the total.
__device__ int scan_array(int32_t* v, int n, int* warp_sums) {
  int running = 0;
  for (int i0 = 0; i0 < n; i0 += kScanThreads) {
    const int i = i0 + threadIdx.x;
    const int x = i < n ? v[i] : 0;
    int tot;
    const int ex = scan_block(x, warp_sums, &tot);
    if (i < n) v[i] = running + ex;
    running += tot;
  }
  return running;
}

__global__ void __launch_bounds__(kScanThreads, 1) hs_scan_kernel(HsParams p) {
  __shared__ int warp_sums[32];
  pdl_wait();
  pdl_trigger();
  const int n_miss = scan_array(p.c.miss, p.n_entry_chunks, warp_sums);
  int n_hit = 0;
  for (int i = threadIdx.x; i < p.n_entry_chunks; i += kScanThreads) n_hit += p.c.hit[i];
  int tot_h;
  scan_block(n_hit, warp_sums, &tot_h);
  const int n_a = scan_array(p.c.a, p.n_lru_chunks, warp_sums);
  if (threadIdx.x == 0) {
    // every requested row must fit: each miss takes a slot not used in this step
    const int overflow = n_miss > n_a;
    p.s.stats[ST_NOT_USED] = n_a;
    if (overflow) atomicOr(p.err, DEV_ERR_CAPACITY);
    p.s.stats[ST_OVERFLOW] = overflow;
    p.s.stats[ST_REQUESTS] = tot_h + n_miss;
    p.s.stats[ST_HITS] = tot_h;
    p.s.stats[ST_MISSES] = overflow ? 0 : n_miss;
    p.s.stats[ST_EVICTED] = 0;
  }
}

__global__ void __launch_bounds__(kThreads) hs_scatter_kernel(HsParams p) {
  __shared__ int warp_sums[32];
  pdl_wait();
  pdl_trigger();
  if (p.s.stats[ST_OVERFLOW]) return;
  const uint32_t step = (uint32_t)p.s.stats[ST_STEP] + 1u;
  const int n_miss = p.s.stats[ST_MISSES];
  const int cap = p.capacity;
  const int n_entries = p.T * p.k;
  if ((int)blockIdx.x < p.n_entry_chunks) {
    // misses in first-request (flat entry) order
    int kinds[kPer];
    int64_t rows[kPer];
    int miss = 0;
    const int f0 = blockIdx.x * kChunk + threadIdx.x * kPer;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      kinds[i] = 0;
      rows[i] = -1;
    }
    if (f0 < n_entries) entry_kinds(p, f0, step, rows, kinds);
#pragma unroll
    for (int i = 0; i < kPer; ++i) miss += kinds[i] == 1;
    int tot;
    int pos = p.c.miss[blockIdx.x] + scan_block(miss, warp_sums, &tot);
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (kinds[i] == 1) p.s.miss_rows[pos++] = (int32_t)rows[i];
  } else {
    const int chunk = blockIdx.x - p.n_entry_chunks;
    const int par = p.s.stats[ST_PARITY] & 1;
    const int32_t* lru = p.s.lru[par];
    int32_t* nxt = p.s.lru[par ^ 1];
    const int n_a = p.s.stats[ST_NOT_USED];
    int slots[kPer], is_a[kPer];
    int a = 0;
    const int i0 = chunk * kChunk + threadIdx.x * kPer;
#pragma unroll
    for (int i = 0; i < kPer; ++i) slots[i] = -1;
    if (i0 < cap) lru_slots(lru, i0, cap, slots);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if ((unsigned)slots[i] >= (unsigned)cap) slots[i] = -1;
      is_a[i] = slots[i] >= 0 && p.s.used[slots[i] >= 0 ? slots[i] : 0] != (int32_t)step;
      a += is_a[i];
    }
    int tot;
    // order: [not-used, not victims] ++ [used] ++ [victims]; a_idx / b_idx count
    // the not-used / used slots before this thread's first one
    int a_idx = p.c.a[chunk] + scan_block(a, warp_sums, &tot);
    int b_idx = i0 - a_idx;
    int evicted = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (slots[i] < 0) continue;
      const int slot = slots[i];
      if (is_a[i]) {
        if (a_idx < n_miss) {
          // victim a_idx receives miss row a_idx (bound in the copy pass); its old row leaves HBM
          const int old = p.s.row_of_slot[slot];
          if (old >= 0) {
            p.s.slot_of_row[old] = -1;
            ++evicted;
          }
          p.s.miss_slots[a_idx] = slot;
          nxt[cap - n_miss + a_idx] = slot;
        } else {
          nxt[a_idx - n_miss] = slot;
        }
        ++a_idx;
      } else {
        nxt[n_a - n_miss + b_idx] = slot;
        ++b_idx;
      }
    }
    int tot_e;
    scan_block(evicted, warp_sums, &tot_e);
    if (threadIdx.x == 0 && tot_e) atomicAdd(p.s.stats + ST_EVICTED, tot_e);
  }
}

__global__ void __launch_bounds__(32 * kCopyWarps) hs_copy_kernel(HsParams p) {
  pdl_wait();
  pdl_trigger();
  const uint32_t step = (uint32_t)p.s.stats[ST_STEP] + 1u;
  const bool overflow = p.s.stats[ST_OVERFLOW] != 0;
  const int a = blockIdx.x * kCopyWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (overflow || a >= p.s.stats[ST_MISSES]) return;
  const int row = p.s.miss_rows[a];
  const int slot = p.s.miss_slots[a];
  if (lane == 0) {
    p.s.row_of_slot[slot] = row;
    p.s.slot_of_row[row] = slot;
    p.s.used[slot] = (int32_t)step;
  }
  const uint4* src = reinterpret_cast<const uint4*>(p.host.base + (int64_t)row * p.host.row_stride);
  uint4* dst = reinterpret_cast<uint4*>(p.slot_pool + (int64_t)slot * p.slot_stride);
  for (int i = lane; i < p.row_elems / 8; i += 32) dst[i] = src[i];
}

__global__ void __launch_bounds__(kThreads) hs_resolve_kernel(HsParams p) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // the step is over: nothing after this kernel in the fetch reads the step or the parity
    p.s.stats[ST_STEP] += 1;
    if (!p.s.stats[ST_OVERFLOW]) p.s.stats[ST_PARITY] ^= 1;
  }
  const int f = blockIdx.x * kThreads + threadIdx.x;
  if (f >= p.T * p.k) return;
  const int t = f / p.k, j = f - t * p.k;
  const int64_t row = entry_row(p, f, false);
  p.slots[(int64_t)t * p.ld_slots + j] = row >= 0 ? p.s.slot_of_row[row] : -1;
}

__global__ void hs_resident_kernel(HsState s, int32_t capacity, int32_t* rows) {
  const int32_t* lru = s.lru[s.stats[ST_PARITY] & 1];
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < capacity; i += gridDim.x * blockDim.x) {
    const int slot = lru[i];
    rows[i] = (unsigned)slot < (unsigned)capacity ? s.row_of_slot[slot] : -1;
  }
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

size_t hisparse_counts_bytes(int64_t entries, int64_t capacity) { return counts_bytes(entries, capacity); }

cudaError_t launch_hisparse_reset(void* state, int32_t capacity, int64_t host_rows, cudaStream_t stream) {
  const HsState s = carve(state, capacity, host_rows);
  const int64_t n = std::max<int64_t>(host_rows, capacity);
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 4096);
  hs_reset_kernel<<<grid, 256, 0, stream>>>(s, capacity, host_rows);
  return cudaGetLastError();
}

cudaError_t launch_hisparse_fetch(const HisparseLaunch& a, cudaStream_t stream) {
  const int64_t n = (int64_t)a.T * a.k;
  HsParams p;
  p.s = carve(a.state, a.capacity, a.host_rows);
  p.c = carve_counts(a.counts, n, a.capacity);
  p.n_entry_chunks = (int32_t)entry_chunks(n);
  p.n_lru_chunks = (int32_t)lru_chunks(a.capacity);
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
  const int entry_grid = (int)((n + kThreads - 1) / kThreads);
  const int chunk_grid = p.n_entry_chunks + p.n_lru_chunks;
  const int max_miss = (int)std::min<int64_t>(n, a.capacity);
  const int copy_grid = std::max(1, (max_miss + kCopyWarps - 1) / kCopyWarps);
  cudaError_t e;
  if ((e = launch_pdl(reinterpret_cast<const void*>(hs_lookup_kernel), entry_grid, kThreads, args, stream))) return e;
  if ((e = launch_pdl(reinterpret_cast<const void*>(hs_count_kernel), chunk_grid, kThreads, args, stream))) return e;
  if ((e = launch_pdl(reinterpret_cast<const void*>(hs_scan_kernel), 1, kScanThreads, args, stream))) return e;
  if ((e = launch_pdl(reinterpret_cast<const void*>(hs_scatter_kernel), chunk_grid, kThreads, args, stream)))
    return e;
  if ((e = launch_pdl(reinterpret_cast<const void*>(hs_copy_kernel), copy_grid, 32 * kCopyWarps, args, stream)))
    return e;
  return launch_pdl(reinterpret_cast<const void*>(hs_resolve_kernel), entry_grid, kThreads, args, stream);
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

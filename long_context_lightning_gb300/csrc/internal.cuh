// internal.cuh -- definitions shared by the kernels and the host launchers of
// the DSA library (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/dsa.h"
#include "ptx.cuh"

namespace dsa {

// Device view of a dsa_cache_t.
struct CacheView {
  const __nv_bfloat16* base;
  int64_t row_stride;
  int64_t num_rows;
  const int64_t* seq_start;
  const int32_t* page_table;
  int64_t pt_stride;
  int32_t page_size;
  int32_t paged;
  int32_t rows;  // positions are pool rows (no sequence addressing)
};

// Pool row of token s of sequence b, or -1 when the page id / row is out of range.
__device__ __forceinline__ int64_t cache_row(const CacheView& c, int b, int64_t s) {
  int64_t row;
  if (c.rows) {
    row = s;
  } else if (c.paged) {
    const int64_t page = s / c.page_size;
    const int64_t phys = __ldg(c.page_table + (int64_t)b * c.pt_stride + page);
    row = phys * c.page_size + (s - page * c.page_size);
    if (phys < 0) return -1;
  } else {
    row = __ldg(c.seq_start + b) + s;
  }
  return (row >= 0 && row < c.num_rows) ? row : -1;
}

// ------------------------------------------------------------------ plan ---
// Per-call plan written to the head of the workspace by plan_kernel:
//   q_seq[T]  sequence of query t
//   q_n[T]    causal context n_t = (p_t + 1) / ratio cache entries (one per token
//             when ratio = 1; 0 when its sequence is malformed)
//   groups    consecutive queries of one sequence scored together by the
//             indexer (G per group): g_info[g] = {b, first query, #queries,
//             n of the group's last query}, g_tile_start[g] = first 128-key
//             work item of group g (prefix sum), g_tile_start[n_groups] = total
//   header    {n_groups, total_items}
struct PlanView {
  int32_t* header;       // [4]
  int32_t* q_seq;        // [T]
  int32_t* q_n;          // [T]
  int4* g_info;          // [T]
  int32_t* g_tile_start; // [T + 1]
};

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline size_t plan_bytes(int64_t T) {
  return align_up(16, 256) + align_up(4 * T, 256) * 2 + align_up(16 * T, 256) + align_up(4 * (T + 1), 256);
}

inline PlanView plan_view(void* ws, int64_t T) {
  char* p = static_cast<char*>(ws);
  PlanView v;
  v.header = reinterpret_cast<int32_t*>(p);
  p += align_up(16, 256);
  v.q_seq = reinterpret_cast<int32_t*>(p);
  p += align_up(4 * T, 256);
  v.q_n = reinterpret_cast<int32_t*>(p);
  p += align_up(4 * T, 256);
  v.g_info = reinterpret_cast<int4*>(p);
  p += align_up(16 * T, 256);
  v.g_tile_start = reinterpret_cast<int32_t*>(p);
  return v;
}

struct PlanParams {
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens_k;
  int32_t B;
  int32_t T;
  int32_t max_seqlen_k;
  int32_t group;        // G queries per indexer group
  int32_t skip_dense_k; // groups whose every query has n <= skip are given no work
  int32_t ratio;        // tokens per cache entry: a query at position p sees (p + 1) / ratio entries
  PlanView plan;
  int* err;
};

constexpr int kIdxTileKeys = 128;  // keys per indexer work item (tcgen05 M)

// Host launchers (each .cu file defines its own).
cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);
// Launch attribute for programmatic dependent launch (kernels call pdl_wait()).
cudaLaunchAttribute pdl_attribute();

struct IndexerLaunch {
  CacheView k;
  const void* q;
  const float* w;
  int32_t H;
  int32_t d;
  int32_t T;
  int32_t group;      // G
  bool keys_once;     // every sequence is one query group: each key tile is read once
  float* scores;
  int64_t ld;
  PlanView plan;
  int* err;
  int num_sms;
};
cudaError_t launch_indexer(const IndexerLaunch& a, cudaStream_t stream);

struct TopkLaunch {
  const float* scores;
  int64_t ld_scores;
  int32_t* idx;
  int64_t ld_idx;
  int32_t k;
  int32_t T;
  int32_t max_n;
  const int32_t* q_n;
  int* err;
  int num_sms;
  // the plan kernel is not the immediately preceding launch: its outputs are
  // complete before this grid starts and may be read before griddepcontrol.wait
  bool plan_early = false;
};
cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t stream);

struct MlaLayerView {
  const __nv_bfloat16* q;
  CacheView kv;
  __nv_bfloat16* out;
  float* lse;
  float scale;
  int32_t H;
};
struct MlaLaunch {
  MlaLayerView layer[DSA_MAX_LAYERS];
  int32_t n_layers;
  int32_t d_qk;
  int32_t d_v;
  const int32_t* idx;
  int64_t ld_idx;
  int32_t k;
  int32_t T;
  int32_t max_n;
  const int32_t* q_seq;
  const int32_t* q_n;
  int* err;
  int num_sms;
  bool plan_early = false;  // as in TopkLaunch
  bool pdl = true;          // programmatic launch after the top-k (off when the stream also waits on an event)
};
cudaError_t launch_sparse_mla(const MlaLaunch& a, cudaStream_t stream);

struct AppendLaunch {
  const void* src;    // bf16 [T, ld_src]
  int64_t ld_src;
  CacheView c;
  int32_t row_elems;  // multiple of 8
  int32_t T;
  int32_t B;
  int32_t max_seqlen_k;
  const int32_t* cu_seqlens_q;  // device [B + 1]
  const int32_t* seq_lens_k;    // device [B]
  int* err;
};
cudaError_t launch_cache_append(const AppendLaunch& a, cudaStream_t stream);

struct HisparseLaunch {
  void* state;
  void* counts;  // hisparse_counts_bytes(T * k, capacity) bytes of the caller's workspace
  int32_t capacity;
  int64_t host_rows;
  int32_t row_elems;
  void* slot_pool;
  int64_t slot_stride;
  CacheView host;
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
size_t hisparse_state_bytes(int64_t capacity, int64_t host_rows);
size_t hisparse_counts_bytes(int64_t entries, int64_t capacity);
cudaError_t launch_hisparse_reset(void* state, int32_t capacity, int64_t host_rows, cudaStream_t stream);
cudaError_t launch_hisparse_fetch(const HisparseLaunch& a, cudaStream_t stream);
cudaError_t launch_hisparse_resident(void* state, int32_t capacity, int64_t host_rows, int32_t* rows,
                                     cudaStream_t stream);
cudaError_t hisparse_read_stats(void* state, int32_t capacity, int64_t host_rows, int32_t* out8, cudaStream_t stream);

// MHA mode: per-head key/value up-projection of a latent pool, and attention
// of every head over the selection (sparse_mha.cu).
struct MhaProjectLaunch {
  const void* c;      // latent pool bf16 [rows, c_stride] (512 latent + 64 rope dims)
  int64_t c_stride;
  int64_t rows;
  int32_t H;
  const void* w_uk;   // bf16 [H, 192, 512]
  const void* w_uv;   // bf16 [H, 256, 512]
  void* k_out;        // bf16 [rows, H, 256]
  void* v_out;        // bf16 [rows, H, 256]
  int* err;
  int num_sms;        // one persistent block per SM
};
struct MhaAttendLaunch {
  PlanView plan;      // groups of up to 128 queries
  CacheView k, v;     // per-head caches (v uses k's addressing)
  const void* q;      // bf16 [T, H, 256]
  const int32_t* idx;
  int64_t ld_idx;
  int32_t k_sel;
  int32_t T;
  int32_t H;
  int32_t W;          // mask words per query
  uint32_t* mask;     // [T, W] (workspace)
  float scale;
  void* out;          // bf16 [T, H, 256]
  float* lse;
  int32_t max_groups;
  int* err;
};
int mha_mask_words(int max_seqlen_k);
cudaError_t launch_mha_project(const MhaProjectLaunch& a, cudaStream_t stream);
cudaError_t launch_mha_attend(const MhaAttendLaunch& a, cudaStream_t stream);

// Largest thread-block cluster (8, or 16 where the device schedules it) for
// kernel `kern` launched with `threads` threads and `smem` bytes of dynamic
// shared memory, on the current device.  Probed once per (device, slot) under
// a lock; non-portable sizes are enabled on that device first.  Returns 0 when
// a CUDA call fails.  `slot` names the kernel variant (kClusterSlot*).
enum { kClusterSlotTopk = 0, kClusterSlotMla0 = 1, kClusterSlotMla1 = 2, kClusterSlots = 4 };
int max_cluster_for(const void* kern, int threads, size_t smem, int slot);
// Cap on the top-k cluster size set by dsa_selftest_topk_max_cluster (0: none).
int topk_cluster_cap();
// Set by dsa_selftest_topk_path(0): the top-k takes the three-pass path only.
bool topk_three_pass_only();

// Tensor-map encoder (driver entry point, resolved once).
CUresult encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                     const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                     CUtensorMapSwizzle swizzle);

}  // namespace dsa

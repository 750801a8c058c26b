// dsa_api.cu -- the C ABI of include/dsa.h: host-side validation, workspace
// layout, tensor-map encoding, the device error word and the launch sequence
// of each entry point.  No call allocates, frees or synchronises (except
// dsa_check_device_error, whose job is to synchronise).
#include <algorithm>
#include <cstring>
#include <mutex>

#include "internal.cuh"

namespace dsa {

__device__ int g_dsa_error_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int* err = nullptr;  // device address of g_dsa_error_word
  int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

dsa_status_t device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.err == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dsa_error_word) != cudaSuccess) return DSA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSA_ERR_CUDA;
    d.err = static_cast<int*>(p);
    d.num_sms = sms;
  }
  *out = d;
  return DSA_OK;
}

// Per-device cluster-size probes of the kernels (see max_cluster_for).
int g_cluster_max[kMaxDevices][kClusterSlots] = {};
int g_topk_cap[kMaxDevices] = {};
bool g_topk_three_pass[kMaxDevices] = {};
std::mutex g_cluster_mu;

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn g_encode = nullptr;
std::once_flag g_encode_once;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

dsa_status_t check_batch(const dsa_batch_t* b) {
  if (b == nullptr) return DSA_ERR_INVALID_ARG;
  if (b->num_seqs < 1 || b->num_seqs > 16384 || b->total_q < 0 || b->max_seqlen_k < 1 || b->max_q_per_seq < 0)
    return DSA_ERR_INVALID_ARG;
  // one grid row per query (per query and layer for the attention): the grid's
  // y extent is at most 65535
  if (b->total_q > DSA_MAX_QUERIES) return DSA_ERR_UNSUPPORTED;
  if (b->total_q > 0 && (b->cu_seqlens_q == nullptr || b->seq_lens_k == nullptr || !aligned4(b->cu_seqlens_q) ||
                         !aligned4(b->seq_lens_k)))
    return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// `max_rows`: the most cache rows (tokens or entries) a sequence of the batch holds.
dsa_status_t check_cache(const dsa_cache_t& c, int row_elems, int64_t max_rows) {
  if (c.base == nullptr || !aligned16(c.base)) return DSA_ERR_INVALID_ARG;
  if (c.row_stride < row_elems || c.row_stride % 8 != 0 || c.num_rows < 1) return DSA_ERR_INVALID_ARG;
  if (c.kind == DSA_CACHE_CONTIGUOUS) {
    if (c.seq_start == nullptr || !aligned8(c.seq_start)) return DSA_ERR_INVALID_ARG;
  } else if (c.kind == DSA_CACHE_PAGED) {
    if (c.page_table == nullptr || !aligned4(c.page_table)) return DSA_ERR_INVALID_ARG;
    if (c.page_size != 64) return DSA_ERR_UNSUPPORTED;
    if (c.page_table_stride < (max_rows + c.page_size - 1) / c.page_size) return DSA_ERR_INVALID_ARG;
  } else if (c.kind == DSA_CACHE_ROWS) {
    // positions are pool rows: nothing to check beyond the pool itself
  } else {
    return DSA_ERR_INVALID_ARG;
  }
  if (c.num_rows > (int64_t)0x7fffffff) return DSA_ERR_UNSUPPORTED;  // TMA row coordinates are int32
  return DSA_OK;
}

CacheView view_of(const dsa_cache_t& c) {
  CacheView v;
  v.base = static_cast<const __nv_bfloat16*>(c.base);
  v.row_stride = c.row_stride;
  v.num_rows = c.num_rows;
  v.seq_start = c.seq_start;
  v.page_table = c.page_table;
  v.pt_stride = c.page_table_stride;
  v.page_size = c.page_size;
  v.paged = c.kind == DSA_CACHE_PAGED;
  v.rows = c.kind == DSA_CACHE_ROWS;
  return v;
}

dsa_status_t check_indexer(const dsa_indexer_t* ix, const dsa_batch_t* b, int ratio = 1) {
  if (ix == nullptr || ix->q == nullptr || ix->w == nullptr || !aligned16(ix->q) || !aligned4(ix->w))
    return DSA_ERR_INVALID_ARG;
  if (ix->k.kind == DSA_CACHE_ROWS) return DSA_ERR_UNSUPPORTED;  // the indexer scores a sequence's tokens
  if (ix->n_heads < 1 || ix->n_heads > 64) return DSA_ERR_UNSUPPORTED;
  if (ix->head_dim != 32 && ix->head_dim != 64 && ix->head_dim != 128) return DSA_ERR_UNSUPPORTED;
  return check_cache(ix->k, ix->head_dim, b->max_seqlen_k / ratio);
}

dsa_status_t check_layer(const dsa_mla_layer_t* l, const dsa_batch_t* b, int ratio = 1) {
  if (l == nullptr || l->q == nullptr || !aligned16(l->q)) return DSA_ERR_INVALID_ARG;
  if (l->n_heads < 1 || l->n_heads > 64) return DSA_ERR_UNSUPPORTED;
  if (!((l->d_qk == 576 && l->d_v == 512) || (l->d_qk == 80 && l->d_v == 64))) return DSA_ERR_UNSUPPORTED;
  if (!(l->scale > 0.f) || l->scale != l->scale) return DSA_ERR_INVALID_ARG;
  return check_cache(l->kv, l->d_qk, b->max_seqlen_k / ratio);
}

// leading dimension of the score matrix: the most entries a query sees, rounded to 4
size_t scores_ld(const dsa_batch_t* b, int ratio = 1) { return align_up((size_t)(b->max_seqlen_k / ratio), 4); }

size_t forward_ws_bytes(const dsa_batch_t* b) {
  return align_up(plan_bytes(b->total_q), 256) + (size_t)b->total_q * scores_ld(b) * sizeof(float);
}

// Plan for this call: q_seq/q_n for every query and the indexer work list.
dsa_status_t run_plan(const dsa_batch_t* b, int group, int skip_dense_k, void* ws, const DeviceInfo& dev,
                      cudaStream_t stream, PlanView* out, int ratio = 1) {
  PlanParams pp;
  pp.cu_seqlens_q = b->cu_seqlens_q;
  pp.seq_lens_k = b->seq_lens_k;
  pp.B = b->num_seqs;
  pp.T = b->total_q;
  pp.max_seqlen_k = b->max_seqlen_k;
  pp.group = group;
  pp.skip_dense_k = skip_dense_k;
  pp.ratio = ratio;
  pp.plan = plan_view(ws, b->total_q);
  pp.err = dev.err;
  *out = pp.plan;
  return launch_plan(pp, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int indexer_group(const dsa_batch_t* b) { return b->max_q_per_seq >= 4 ? 4 : 1; }

dsa_status_t launch_indexer_call(const dsa_batch_t* b, const dsa_indexer_t* ix, float* scores, int64_t ld,
                                 const PlanView& plan, const DeviceInfo& dev, cudaStream_t stream) {
  IndexerLaunch a;
  a.k = view_of(ix->k);
  a.q = ix->q;
  a.w = ix->w;
  a.H = ix->n_heads;
  a.d = ix->head_dim;
  a.T = b->total_q;
  a.group = indexer_group(b);
  a.keys_once = b->max_q_per_seq <= a.group;
  a.scores = scores;
  a.ld = ld;
  a.plan = plan;
  a.err = dev.err;
  a.num_sms = dev.num_sms;
  return launch_indexer(a, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status_t launch_topk_call(const dsa_batch_t* b, const float* scores, int64_t ld, int32_t k, int32_t* idx,
                              int64_t ld_idx, const PlanView& plan, const DeviceInfo& dev, cudaStream_t stream,
                              bool plan_early = false, int ratio = 1) {
  TopkLaunch a;
  a.scores = scores;
  a.ld_scores = ld;
  a.idx = idx;
  a.ld_idx = ld_idx;
  a.k = k;
  a.T = b->total_q;
  a.max_n = std::max(1, b->max_seqlen_k / ratio);
  a.q_n = plan.q_n;
  a.err = dev.err;
  a.num_sms = dev.num_sms;
  a.plan_early = plan_early;
  return launch_topk(a, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status_t launch_mla_call(const dsa_batch_t* b, int n_layers, const dsa_mla_layer_t* layers,
                             void* const* outs, float* const* lses, const int32_t* idx, int64_t ld_idx, int32_t k,
                             const PlanView& plan, const DeviceInfo& dev, cudaStream_t stream,
                             bool plan_early = false, int ratio = 1, bool pdl = true) {
  MlaLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.pdl = pdl;
  for (int l = 0; l < n_layers; ++l) {
    a.layer[l].q = static_cast<const __nv_bfloat16*>(layers[l].q);
    a.layer[l].kv = view_of(layers[l].kv);
    a.layer[l].out = static_cast<__nv_bfloat16*>(outs[l]);
    a.layer[l].lse = lses ? lses[l] : nullptr;
    a.layer[l].scale = layers[l].scale;
    a.layer[l].H = layers[l].n_heads;
  }
  a.n_layers = n_layers;
  a.d_qk = layers[0].d_qk;
  a.d_v = layers[0].d_v;
  a.idx = idx;
  a.ld_idx = ld_idx;
  a.k = k;
  a.T = b->total_q;
  a.max_n = std::max(1, b->max_seqlen_k / ratio);
  a.q_seq = plan.q_seq;
  a.q_n = plan.q_n;
  a.err = dev.err;
  a.num_sms = dev.num_sms;
  a.plan_early = plan_early;
  return launch_sparse_mla(a, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

int max_cluster_for(const void* kern, int threads, size_t smem, int slot) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kClusterSlots)
    return 0;
  std::lock_guard<std::mutex> lock(g_cluster_mu);
  int& m = g_cluster_max[dev][slot];
  if (m == 0) {
    // function attributes are per device: allow non-portable sizes on this one
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return 0;
    int best = 8;
    cudaLaunchConfig_t probe = {};
    probe.gridDim = dim3(16, 1, 1);
    probe.blockDim = dim3(threads, 1, 1);
    probe.dynamicSmemBytes = smem;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 16;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    probe.attrs = &at;
    probe.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &probe) == cudaSuccess && nclusters > 0) best = 16;
    cudaGetLastError();  // a refused probe leaves no sticky error behind
    m = best;
  }
  return m;
}

bool topk_three_pass_only() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_cluster_mu);
  return g_topk_three_pass[dev];
}

int topk_cluster_cap() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_cluster_mu);
  return g_topk_cap[dev];
}

CUresult encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                     const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                     CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeFn>(fn);
  });
  if (g_encode == nullptr) return CUDA_ERROR_NOT_FOUND;
  cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  return g_encode(map, dtype, rank, const_cast<void*>(base), reinterpret_cast<const cuuint64_t*>(dims),
                  reinterpret_cast<const cuuint64_t*>(strides_bytes), reinterpret_cast<const cuuint32_t*>(box),
                  estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// ------------------------------------------------------------- self-tests ---
namespace {

// One 128 x 64 tile through the same descriptors the kernels build.  With
// sw64 the operands are K-major in 64-byte-swizzled atoms, two K-blocks of 32.
__global__ void __launch_bounds__(128, 1)
    selftest_mma_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B, float* D, int a_mn, int b_mn, int sw64,
                        int a_tmem, int* err) {
  __shared__ __align__(1024) uint8_t sa[128 * 128];  // 16 KB
  __shared__ __align__(1024) uint8_t sb[64 * 128];   // 8 KB
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // stage A [128 x 64] (m, k)
  for (int i = tid; i < 128 * 64; i += 128) {
    const int m = i / 64, k = i % 64;
    uint32_t off;
    if (sw64) {          // K-block k/32 of [128 rows x 64 bytes]
      const int kb = k / 32, kk = k % 32;
      off = kb * 8192 + m * 64 + (((kk / 8) ^ ((m >> 1) & 3)) << 4) + (kk % 8) * 2;
    } else if (!a_mn) {  // K-major: row m, 64 k per row
      off = m * 128 + (((k / 8) ^ (m & 7)) << 4) + (k % 8) * 2;
    } else {             // MN-major: two 64-wide m blocks of 64 k-rows, 8 KB apart
      const int mb = m / 64, mm = m % 64;
      off = mb * 8192 + k * 128 + (((mm / 8) ^ (k & 7)) << 4) + (mm % 8) * 2;
    }
    *reinterpret_cast<__nv_bfloat16*>(sa + off) = A[i];
  }
  for (int i = tid; i < 64 * 64; i += 128) {
    const int n = i / 64, k = i % 64;
    uint32_t off;
    if (sw64) {
      const int kb = k / 32, kk = k % 32;
      off = kb * 4096 + n * 64 + (((kk / 8) ^ ((n >> 1) & 3)) << 4) + (kk % 8) * 2;
    } else if (!b_mn) {
      off = n * 128 + (((k / 8) ^ (n & 7)) << 4) + (k % 8) * 2;
    } else {
      off = k * 128 + (((n / 8) ^ (k & 7)) << 4) + (n % 8) * 2;
    }
    *reinterpret_cast<__nv_bfloat16*>(sb + off) = B[i];
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(&tslot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  if (a_tmem) {
    // A row m into lane m, columns 64..95: element pairs (2c, 2c+1) of the row in column c
    const int m = warp * 32 + lane;
    uint32_t r[32];
    for (int c = 0; c < 32; ++c) {
      const uint32_t lo = __bfloat16_as_ushort(A[m * 64 + 2 * c]), hi = __bfloat16_as_ushort(A[m * 64 + 2 * c + 1]);
      r[c] = lo | (hi << 16);
    }
    tmem_st32(tmem + ((uint32_t)(warp * 32) << 16) + 64, r);
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (tid == 0) {
    const uint32_t idesc = mma_idesc_bf16(128, 64, a_mn != 0, b_mn != 0);
    for (int ks = 0; ks < 4; ++ks) {
      uint64_t ad, bd;
      if (a_tmem) {
        bd = b_mn ? smem_desc_sw128(smem_u32(sb) + ks * 2048, 8192, 1024)
                  : smem_desc_sw128(smem_u32(sb) + ks * 32, 16, 1024);
        mma_bf16_ts(tmem, tmem + 64 + ks * 8, bd, idesc, ks != 0);
        continue;
      }
      if (sw64) {
        ad = smem_desc_sw64(smem_u32(sa) + (ks / 2) * 8192 + (ks % 2) * 32, 512);
        bd = smem_desc_sw64(smem_u32(sb) + (ks / 2) * 4096 + (ks % 2) * 32, 512);
      } else {
        ad = a_mn ? smem_desc_sw128(smem_u32(sa) + ks * 2048, 8192, 1024)
                  : smem_desc_sw128(smem_u32(sa) + ks * 32, 16, 1024);
        bd = b_mn ? smem_desc_sw128(smem_u32(sb) + ks * 2048, 8192, 1024)
                  : smem_desc_sw128(smem_u32(sb) + ks * 32, 16, 1024);
      }
      mma_bf16(tmem, ad, bd, idesc, ks != 0);
    }
    mma_commit(smem_u32(&bar));
  }
  __syncwarp();
  mbar_wait(smem_u32(&bar), 0, &abort_flag, err);
  tc_fence_after();
  const int row = warp * 32 + lane;
  for (int c = 0; c < 4; ++c) {
    uint32_t r[16];
    tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c * 16, r);
    tmem_wait_ld();
    for (int j = 0; j < 16; ++j) D[row * 64 + c * 16 + j] = __uint_as_float(r[j]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Waits on a barrier nobody arrives at; the bounded wait gives up and reports.
__global__ void selftest_timeout_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(smem_u32(&bar), 0)) return;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, DEV_ERR_TIMEOUT);
      return;
    }
  }
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: null pointer, misalignment or inconsistent sizes";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: sizes outside the supported set";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace missing or too small";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: a CUDA call or launch failed";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT: a bounded device-side wait ran out";
    case DSA_ERR_BAD_INDEX: return "DSA_ERR_BAD_INDEX: a device-side length, page id or index was out of range";
    case DSA_ERR_CAPACITY: return "DSA_ERR_CAPACITY: a device-side capacity was exceeded";
  }
  return "DSA_ERR_UNKNOWN";
}

dsa_status_t dsa_check_device_error(cudaStream_t stream) {
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSA_ERR_CUDA;
  int word = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_dsa_error_word, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_dsa_error_word, &zero, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  if (word & DEV_ERR_TIMEOUT) return DSA_ERR_TIMEOUT;
  if (word & DEV_ERR_BAD_INDEX) return DSA_ERR_BAD_INDEX;
  if (word & DEV_ERR_CAPACITY) return DSA_ERR_CAPACITY;
  return DSA_OK;
}

size_t dsa_workspace_size(const dsa_batch_t* batch, int32_t topk) {
  if (check_batch(batch) != DSA_OK || topk < 0 || topk > DSA_MAX_TOPK) return 0;
  return forward_ws_bytes(batch);
}

dsa_status_t dsa_indexer_scores(const dsa_batch_t* batch, const dsa_indexer_t* indexer, int32_t skip_dense_k,
                                float* scores, int64_t ld_scores, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
  dsa_status_t s = check_batch(batch);
  if (s != DSA_OK) return s;
  if ((s = check_indexer(indexer, batch)) != DSA_OK) return s;
  if (scores == nullptr || !aligned16(scores) || ld_scores < batch->max_seqlen_k || ld_scores % 4 != 0 ||
      skip_dense_k < 0)
    return DSA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < plan_bytes(batch->total_q))
    return DSA_ERR_WORKSPACE;
  if (batch->total_q == 0) return DSA_OK;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  PlanView plan;
  if ((s = run_plan(batch, indexer_group(batch), skip_dense_k, workspace, dev, stream, &plan)) != DSA_OK) return s;
  return launch_indexer_call(batch, indexer, scores, ld_scores, plan, dev, stream);
}

dsa_status_t dsa_topk(const dsa_batch_t* batch, const float* scores, int64_t ld_scores, int32_t topk, int32_t* idx,
                      int64_t ld_idx, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  dsa_status_t s = check_batch(batch);
  if (s != DSA_OK) return s;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (scores == nullptr || !aligned16(scores) || ld_scores < batch->max_seqlen_k || ld_scores % 4 != 0)
    return DSA_ERR_INVALID_ARG;
  if (idx == nullptr || !aligned4(idx) || ld_idx < topk) return DSA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < plan_bytes(batch->total_q))
    return DSA_ERR_WORKSPACE;
  if (batch->total_q == 0) return DSA_OK;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  PlanView plan;
  if ((s = run_plan(batch, 1, 0, workspace, dev, stream, &plan)) != DSA_OK) return s;
  return launch_topk_call(batch, scores, ld_scores, topk, idx, ld_idx, plan, dev, stream);
}

dsa_status_t dsa_sparse_mla_fwd(const dsa_batch_t* batch, const dsa_mla_layer_t* layer, const int32_t* idx,
                                int64_t ld_idx, int32_t topk, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  dsa_status_t s = check_batch(batch);
  if (s != DSA_OK) return s;
  if ((s = check_layer(layer, batch)) != DSA_OK) return s;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (idx == nullptr || !aligned4(idx) || ld_idx < topk) return DSA_ERR_INVALID_ARG;
  if (out == nullptr || !aligned16(out) || (lse != nullptr && !aligned4(lse))) return DSA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < plan_bytes(batch->total_q))
    return DSA_ERR_WORKSPACE;
  if (batch->total_q == 0) return DSA_OK;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  PlanView plan;
  if ((s = run_plan(batch, 1, 0, workspace, dev, stream, &plan)) != DSA_OK) return s;
  void* outs[1] = {out};
  float* lses[1] = {lse};
  return launch_mla_call(batch, 1, layer, outs, lses, idx, ld_idx, topk, plan, dev, stream);
}

}  // extern "C"

namespace dsa {
namespace {
// indexer -> top-k -> sparse MLA over cache entries of `ratio` tokens (1: tokens)
dsa_status_t forward_impl(const dsa_batch_t* batch, int ratio, const dsa_indexer_t* indexer, int32_t topk,
                          int32_t n_layers, const dsa_mla_layer_t* layers, int32_t* idx, int64_t ld_idx,
                          void* const* outs, float* const* lses, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream, cudaEvent_t const* marks, cudaEvent_t mla_ready = nullptr,
                          cudaEvent_t topk_done = nullptr) {
  dsa_status_t s = check_batch(batch);
  if (s != DSA_OK) return s;
  if (ratio < 1 || ratio > batch->max_seqlen_k) return DSA_ERR_INVALID_ARG;
  if ((s = check_indexer(indexer, batch, ratio)) != DSA_OK) return s;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (n_layers < 1 || n_layers > DSA_MAX_LAYERS || layers == nullptr || outs == nullptr) return DSA_ERR_INVALID_ARG;
  if ((int64_t)batch->total_q * n_layers > DSA_MAX_QUERIES) return DSA_ERR_UNSUPPORTED;
  for (int l = 0; l < n_layers; ++l) {
    if ((s = check_layer(&layers[l], batch, ratio)) != DSA_OK) return s;
    if (layers[l].d_qk != layers[0].d_qk || layers[l].d_v != layers[0].d_v) return DSA_ERR_UNSUPPORTED;
    if (outs[l] == nullptr || !aligned16(outs[l])) return DSA_ERR_INVALID_ARG;
    if (lses != nullptr && lses[l] != nullptr && !aligned4(lses[l])) return DSA_ERR_INVALID_ARG;
  }
  if (idx == nullptr || !aligned4(idx) || ld_idx < topk) return DSA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < forward_ws_bytes(batch))
    return DSA_ERR_WORKSPACE;
  if (batch->total_q == 0) return DSA_OK;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  auto mark = [&](int i) { return marks == nullptr || cudaEventRecord(marks[i], stream) == cudaSuccess; };
  if (!mark(0)) return DSA_ERR_CUDA;
  PlanView plan;
  if ((s = run_plan(batch, indexer_group(batch), topk, workspace, dev, stream, &plan, ratio)) != DSA_OK) return s;
  if (!mark(1)) return DSA_ERR_CUDA;
  float* scores = reinterpret_cast<float*>(static_cast<char*>(workspace) + align_up(plan_bytes(batch->total_q), 256));
  const int64_t ld = (int64_t)scores_ld(batch, ratio);
  if ((s = launch_indexer_call(batch, indexer, scores, ld, plan, dev, stream)) != DSA_OK) return s;
  if (!mark(2)) return DSA_ERR_CUDA;
  // the plan kernel ran two launches before the top-k and three before the MLA
  if ((s = launch_topk_call(batch, scores, ld, topk, idx, ld_idx, plan, dev, stream, true, ratio)) != DSA_OK)
    return s;
  if (!mark(3)) return DSA_ERR_CUDA;
  if (topk_done != nullptr && cudaEventRecord(topk_done, stream) != cudaSuccess) return DSA_ERR_CUDA;
  if (mla_ready != nullptr && cudaStreamWaitEvent(stream, mla_ready, 0) != cudaSuccess) return DSA_ERR_CUDA;
  // a launch that also waits on the caller's event is an ordinary one: a
  // programmatic edge may not join another stream's work in a captured graph
  if ((s = launch_mla_call(batch, n_layers, layers, outs, lses, idx, ld_idx, topk, plan, dev, stream, true,
                           ratio, mla_ready == nullptr)) != DSA_OK)
    return s;
  return mark(4) ? DSA_OK : DSA_ERR_CUDA;
}
}  // namespace
}  // namespace dsa

extern "C" {

dsa_status_t dsa_forward_marked(const dsa_batch_t* batch, const dsa_indexer_t* indexer, int32_t topk,
                                int32_t n_layers, const dsa_mla_layer_t* layers, int32_t* idx, int64_t ld_idx,
                                void* const* outs, float* const* lses, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream, cudaEvent_t const* marks) {
  return forward_impl(batch, 1, indexer, topk, n_layers, layers, idx, ld_idx, outs, lses, workspace,
                      workspace_bytes, stream, marks);
}

dsa_status_t dsa_forward_compressed(const dsa_batch_t* batch, int32_t compress_ratio, const dsa_indexer_t* indexer,
                                    int32_t topk, int32_t n_layers, const dsa_mla_layer_t* layers, int32_t* idx,
                                    int64_t ld_idx, void* const* outs, float* const* lses, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream, cudaEvent_t const* marks) {
  return forward_impl(batch, compress_ratio, indexer, topk, n_layers, layers, idx, ld_idx, outs, lses, workspace,
                      workspace_bytes, stream, marks);
}

dsa_status_t dsa_forward_overlapped(const dsa_batch_t* batch, const dsa_indexer_t* indexer, int32_t topk,
                                    int32_t n_layers, const dsa_mla_layer_t* layers, int32_t* idx, int64_t ld_idx,
                                    void* const* outs, float* const* lses, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream, cudaEvent_t mla_ready, cudaEvent_t topk_done) {
  return forward_impl(batch, 1, indexer, topk, n_layers, layers, idx, ld_idx, outs, lses, workspace,
                      workspace_bytes, stream, nullptr, mla_ready, topk_done);
}

dsa_status_t dsa_forward(const dsa_batch_t* batch, const dsa_indexer_t* indexer, int32_t topk, int32_t n_layers,
                         const dsa_mla_layer_t* layers, int32_t* idx, int64_t ld_idx, void* const* outs,
                         float* const* lses, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return dsa_forward_marked(batch, indexer, topk, n_layers, layers, idx, ld_idx, outs, lses, workspace,
                            workspace_bytes, stream, nullptr);
}

}  // extern "C"

// ------------------------------------------- sparse MLA without a workspace ---
// Some callers cannot hand the library any device memory beyond their inputs
// and outputs: a plugin interface that passes only tensor pointers, or an
// engine whose device memory is entirely claimed by its own pool, so a
// cudaMalloc at call time would fail (or stall the device).  For them the
// per-call plan of dsa_sparse_mla_fwd lives in this file-scope array instead
// of a workspace.  Every GPU that loads the library holds it until exit.
namespace dsa {
namespace {

constexpr int kNoAllocMaxQ = DSA_NOALLOC_MAX_QUERIES;
constexpr size_t kNoAllocScratchBytes = align_up(16, 256) + 2 * align_up(4 * (size_t)kNoAllocMaxQ, 256) +
                                        align_up(16 * (size_t)kNoAllocMaxQ, 256) +
                                        align_up(4 * (size_t)(kNoAllocMaxQ + 1), 256);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_noalloc_ptr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device
std::mutex g_noalloc_mu;

// Once per device, with that device current: the host-side name of the array
// is only a stand-in, so the kernels get the address the runtime reports.
dsa_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" {

dsa_status_t dsa_sparse_mla_fwd_noalloc(const dsa_batch_t* batch, const dsa_mla_layer_t* layer, const int32_t* idx,
                                        int64_t ld_idx, int32_t topk, void* out, float* lse, cudaStream_t stream) {
  dsa_status_t s = check_batch(batch);
  if (s != DSA_OK) return s;
  if (batch->total_q > DSA_NOALLOC_MAX_QUERIES) return DSA_ERR_UNSUPPORTED;  // beyond the static scratch
  if (plan_bytes(batch->total_q) > kNoAllocScratchBytes) return DSA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if ((s = noalloc_scratch(&scratch)) != DSA_OK) return s;
  // The plan kernel rewrites every entry the attention kernel reads, so the
  // previous call's contents need no clearing.
  return dsa_sparse_mla_fwd(batch, layer, idx, ld_idx, topk, out, lse, scratch, kNoAllocScratchBytes, stream);
}

dsa_status_t dsa_selftest_mma(const void* a, const void* b, float* d, int32_t a_mn_major, int32_t b_mn_major,
                              int32_t swizzle_bytes, cudaStream_t stream) {
  if (a == nullptr || b == nullptr || d == nullptr) return DSA_ERR_INVALID_ARG;
  if (swizzle_bytes != 128 && swizzle_bytes != 64 && swizzle_bytes != 0) return DSA_ERR_INVALID_ARG;
  if (swizzle_bytes == 64 && (a_mn_major || b_mn_major)) return DSA_ERR_UNSUPPORTED;
  if (swizzle_bytes == 0 && a_mn_major) return DSA_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  selftest_mma_kernel<<<1, 128, 0, stream>>>(static_cast<const __nv_bfloat16*>(a),
                                              static_cast<const __nv_bfloat16*>(b), d, a_mn_major, b_mn_major,
                                              swizzle_bytes == 64, swizzle_bytes == 0, dev.err);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status_t dsa_cache_append(const dsa_batch_t* batch, const void* rows, int64_t ld_rows, int32_t row_elems,
                              const dsa_cache_t* cache, cudaStream_t stream) {
  dsa_status_t s = check_batch(batch);
  if (s != DSA_OK) return s;
  if (cache == nullptr || rows == nullptr || !aligned16(rows)) return DSA_ERR_INVALID_ARG;
  if (row_elems < 8 || row_elems % 8 != 0 || ld_rows < row_elems || ld_rows % 8 != 0) return DSA_ERR_INVALID_ARG;
  if ((s = check_cache(*cache, row_elems, batch->max_seqlen_k)) != DSA_OK) return s;
  if (batch->total_q == 0) return DSA_OK;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  AppendLaunch a;
  a.src = rows;
  a.ld_src = ld_rows;
  a.c = view_of(*cache);
  a.row_elems = row_elems;
  a.T = batch->total_q;
  a.B = batch->num_seqs;
  a.max_seqlen_k = batch->max_seqlen_k;
  a.cu_seqlens_q = batch->cu_seqlens_q;
  a.seq_lens_k = batch->seq_lens_k;
  a.err = dev.err;
  return launch_cache_append(a, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

size_t dsa_hisparse_state_bytes(int32_t capacity, int64_t host_rows) {
  if (capacity < 1 || host_rows < 1) return 0;
  return hisparse_state_bytes(capacity, host_rows);
}

size_t dsa_hisparse_workspace_size(const dsa_batch_t* batch, int32_t topk, int32_t capacity) {
  if (check_batch(batch) != DSA_OK || topk < 1 || topk > DSA_MAX_TOPK || capacity < 1) return 0;
  return plan_bytes(batch->total_q) + hisparse_counts_bytes((int64_t)batch->total_q * topk, capacity);
}

static dsa_status_t check_hisparse(const dsa_hisparse_t* hs) {
  if (hs == nullptr || hs->capacity < 1 || hs->host_rows < 1 || hs->host_rows > (int64_t)0x7fffffff)
    return DSA_ERR_INVALID_ARG;
  if (hs->row_elems < 8 || hs->row_elems % 8 != 0 || hs->slot_stride < hs->row_elems || hs->slot_stride % 8 != 0)
    return DSA_ERR_INVALID_ARG;
  if (hs->slot_pool == nullptr || !aligned16(hs->slot_pool) || hs->state == nullptr || !aligned16(hs->state))
    return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

dsa_status_t dsa_hisparse_reset(const dsa_hisparse_t* hs, cudaStream_t stream) {
  dsa_status_t s = check_hisparse(hs);
  if (s != DSA_OK) return s;
  return launch_hisparse_reset(hs->state, hs->capacity, hs->host_rows, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status_t dsa_hisparse_fetch(const dsa_hisparse_t* hs, const dsa_batch_t* batch, const dsa_cache_t* host_cache,
                                const int32_t* idx, int64_t ld_idx, int32_t topk, int32_t* slots, int64_t ld_slots,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  dsa_status_t s = check_batch(batch);
  if (s != DSA_OK) return s;
  if ((s = check_hisparse(hs)) != DSA_OK) return s;
  if (host_cache == nullptr || host_cache->kind == DSA_CACHE_ROWS || host_cache->num_rows != hs->host_rows)
    return DSA_ERR_INVALID_ARG;
  if ((s = check_cache(*host_cache, hs->row_elems, batch->max_seqlen_k)) != DSA_OK) return s;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (idx == nullptr || !aligned4(idx) || ld_idx < topk) return DSA_ERR_INVALID_ARG;
  if (slots == nullptr || !aligned4(slots) || ld_slots < topk) return DSA_ERR_INVALID_ARG;
  if ((int64_t)batch->total_q * topk > (int64_t)0x7fffffff) return DSA_ERR_UNSUPPORTED;
  if (workspace == nullptr || !aligned16(workspace) ||
      workspace_bytes < dsa_hisparse_workspace_size(batch, topk, hs->capacity))
    return DSA_ERR_WORKSPACE;
  if (batch->total_q == 0) return DSA_OK;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  PlanView plan;
  if ((s = run_plan(batch, 1, 0, workspace, dev, stream, &plan)) != DSA_OK) return s;
  // the host pool must be memory the device can read: pinned or registered
  // host memory (its device address is used), or device / managed memory
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, host_cache->base) != cudaSuccess) {
    cudaGetLastError();
    return DSA_ERR_INVALID_ARG;
  }
  if (attr.type == cudaMemoryTypeUnregistered || attr.devicePointer == nullptr) return DSA_ERR_INVALID_ARG;
  dsa_cache_t host = *host_cache;
  host.base = attr.devicePointer;
  HisparseLaunch a;
  a.state = hs->state;
  a.counts = static_cast<char*>(workspace) + plan_bytes(batch->total_q);
  a.capacity = hs->capacity;
  a.host_rows = hs->host_rows;
  a.row_elems = hs->row_elems;
  a.slot_pool = hs->slot_pool;
  a.slot_stride = hs->slot_stride;
  a.host = view_of(host);
  a.idx = idx;
  a.ld_idx = ld_idx;
  a.k = topk;
  a.T = batch->total_q;
  a.q_seq = plan.q_seq;
  a.q_n = plan.q_n;
  a.slots = slots;
  a.ld_slots = ld_slots;
  a.err = dev.err;
  return launch_hisparse_fetch(a, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status_t dsa_hisparse_resident(const dsa_hisparse_t* hs, int32_t* rows, cudaStream_t stream) {
  dsa_status_t s = check_hisparse(hs);
  if (s != DSA_OK) return s;
  if (rows == nullptr || !aligned4(rows)) return DSA_ERR_INVALID_ARG;
  return launch_hisparse_resident(hs->state, hs->capacity, hs->host_rows, rows, stream) == cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}

dsa_status_t dsa_hisparse_stats(const dsa_hisparse_t* hs, int32_t* stats, cudaStream_t stream) {
  dsa_status_t s = check_hisparse(hs);
  if (s != DSA_OK) return s;
  if (stats == nullptr) return DSA_ERR_INVALID_ARG;
  return hisparse_read_stats(hs->state, hs->capacity, hs->host_rows, stats, stream) == cudaSuccess ? DSA_OK
                                                                                                  : DSA_ERR_CUDA;
}

dsa_status_t dsa_mha_project(const void* latent, int64_t latent_stride, int64_t rows, int32_t n_heads,
                             const void* w_uk, const void* w_uv, void* k_out, void* v_out, cudaStream_t stream) {
  if (rows < 0 || rows > (int64_t)0x7fffffff || n_heads < 1 || n_heads > DSA_MHA_MAX_HEADS)
    return DSA_ERR_INVALID_ARG;
  if (latent_stride < DSA_MHA_LATENT + DSA_MHA_ROPE || latent_stride % 8 != 0) return DSA_ERR_INVALID_ARG;
  const void* ptrs[5] = {latent, w_uk, w_uv, k_out, v_out};
  for (const void* q : ptrs)
    if (q == nullptr || !aligned16(q)) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  MhaProjectLaunch a;
  a.c = latent;
  a.c_stride = latent_stride;
  a.rows = rows;
  a.H = n_heads;
  a.w_uk = w_uk;
  a.w_uv = w_uv;
  a.k_out = k_out;
  a.v_out = v_out;
  a.err = dev.err;
  a.num_sms = dev.num_sms;
  return launch_mha_project(a, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

static size_t mha_mask_bytes(const dsa_batch_t* b) {
  return align_up((size_t)b->total_q * mha_mask_words(b->max_seqlen_k) * 4, 256);
}

size_t dsa_mha_workspace_size(const dsa_batch_t* batch) {
  if (check_batch(batch) != DSA_OK || batch->max_seqlen_k > DSA_MHA_MAX_CONTEXT) return 0;
  return plan_bytes(batch->total_q) + mha_mask_bytes(batch);
}

dsa_status_t dsa_sparse_mha_fwd(const dsa_batch_t* batch, const dsa_mha_layer_t* layer, const int32_t* idx,
                                int64_t ld_idx, int32_t topk, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  dsa_status_t s = check_batch(batch);
  if (s != DSA_OK) return s;
  if (layer == nullptr || layer->q == nullptr || !aligned16(layer->q)) return DSA_ERR_INVALID_ARG;
  if (layer->head_dim != DSA_MHA_HEAD_DIM || layer->v_head_dim != DSA_MHA_HEAD_DIM) return DSA_ERR_UNSUPPORTED;
  if (layer->n_heads < 1 || layer->n_heads > DSA_MHA_MAX_HEADS) return DSA_ERR_UNSUPPORTED;
  if (!(layer->scale > 0.f)) return DSA_ERR_INVALID_ARG;  // a softmax scale: positive (and not NaN)
  if (batch->max_seqlen_k > DSA_MHA_MAX_CONTEXT) return DSA_ERR_UNSUPPORTED;
  const dsa_cache_t& kc = layer->k;
  const dsa_cache_t& vc = layer->v;
  if (kc.kind == DSA_CACHE_ROWS || vc.kind != kc.kind || vc.num_rows != kc.num_rows ||
      vc.seq_start != kc.seq_start || vc.page_table != kc.page_table ||
      vc.page_table_stride != kc.page_table_stride)
    return DSA_ERR_INVALID_ARG;
  const int row_elems = layer->n_heads * DSA_MHA_HEAD_DIM;
  if ((s = check_cache(kc, row_elems, batch->max_seqlen_k)) != DSA_OK) return s;
  if ((s = check_cache(vc, row_elems, batch->max_seqlen_k)) != DSA_OK) return s;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (idx == nullptr || !aligned4(idx) || ld_idx < topk) return DSA_ERR_INVALID_ARG;
  if (out == nullptr || !aligned16(out) || (lse != nullptr && !aligned4(lse))) return DSA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < dsa_mha_workspace_size(batch))
    return DSA_ERR_WORKSPACE;
  if (batch->total_q == 0) return DSA_OK;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  PlanView plan;
  constexpr int kGroup = 128;  // queries per attention block
  if ((s = run_plan(batch, kGroup, 0, workspace, dev, stream, &plan)) != DSA_OK) return s;
  MhaAttendLaunch a;
  a.plan = plan;
  a.k = view_of(kc);
  a.v = view_of(vc);
  a.q = layer->q;
  a.idx = idx;
  a.ld_idx = ld_idx;
  a.k_sel = topk;
  a.T = batch->total_q;
  a.H = layer->n_heads;
  a.W = mha_mask_words(batch->max_seqlen_k);
  a.mask = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + plan_bytes(batch->total_q));
  a.scale = layer->scale;
  a.out = out;
  a.lse = lse;
  // groups never straddle sequences: at most one partial group per sequence
  a.max_groups = (batch->total_q + kGroup - 1) / kGroup + batch->num_seqs;
  a.err = dev.err;
  return launch_mha_attend(a, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status_t dsa_selftest_topk_max_cluster(int32_t max_cluster) {
  if (max_cluster != 0 && max_cluster != 1 && max_cluster != 2 && max_cluster != 4 && max_cluster != 8 &&
      max_cluster != 16)
    return DSA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_cluster_mu);
  g_topk_cap[dev] = max_cluster;
  return DSA_OK;
}

dsa_status_t dsa_selftest_topk_path(int32_t candidates) {
  if (candidates != 0 && candidates != 1) return DSA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_cluster_mu);
  g_topk_three_pass[dev] = candidates == 0;
  return DSA_OK;
}

dsa_status_t dsa_selftest_timeout(int32_t limit_ms, cudaStream_t stream) {
  if (limit_ms < 1 || limit_ms > 10000) return DSA_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (device_info(&dev) != DSA_OK) return DSA_ERR_CUDA;
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(dev.err, (uint64_t)limit_ms * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // extern "C"

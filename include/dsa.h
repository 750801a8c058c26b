/*
 * dsa.h -- C ABI of the DeepSeek Sparse Attention (DSA) forward path on one
 * GB300 GPU (sm_103a).
 *
 * The path has three steps, each exported on its own and fused in dsa_forward:
 *
 *   1. lightning indexer: for query token t and past token s <= p_t,
 *        I[t, s] = sum_h w[t, h] * max(0, q_I[t, h, :] . k_I[s, :])
 *      ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it works /
 *      Model, lightning-indexer bullet: a down-projected ReLU dot product summed
 *      with weights across heads; "DeepSeek Sparse Attention", In the code
 *      table: ReLU(q.k) scores summed with weights, index_n_heads / index_head_dim).
 *   2. top-k: the k past tokens with the largest I[t, .]; when the causal
 *      context holds at most k tokens, all of them ("How GLM5.3 ...", Model,
 *      sparse-MLA bullet: top-k 2048, attention below 2K stays dense).  Equal
 *      scores go to the lower position; -0.0 equals +0.0.
 *   3. sparse MLA in MQA mode: every attention head attends with softmax over
 *      the selected latent rows only; all heads read the same 576-dim latent
 *      row of a token, the value is its first d_v dims ("How GLM5.3 ...",
 *      Model, sparse-MLA bullet).
 *   IndexShare: one indexer + top-k serves a group of layers, each attending
 *   over the same index set with its own query and latent cache ("How GLM5.3
 *   ...", How it works / IndexShare: every 4 DSA layers share one indexer and
 *   the top-k indices are cached for the shared layers).
 *
 * Conventions shared by every call
 *   - All pointers named "device" are CUDA device pointers of the current
 *     device; the caller allocates, owns and frees every buffer.  The library
 *     never allocates, frees or synchronises inside a compute call; every
 *     compute call is asynchronous on `stream` and launches only kernels.
 *   - Data types are fixed: bf16 (raw 16-bit storage, `const void*`) for
 *     queries, caches and attention outputs; fp32 for head weights, scores and
 *     LSE; int32 for lengths, page tables and selected positions.
 *   - Every device pointer must be 16-byte aligned; every row stride is in
 *     elements and must make rows 16-byte aligned.
 *   - Ragged batches: sequence b has seq_lens_k[b] cached tokens, and its
 *     queries are its LAST cu_seqlens_q[b+1]-cu_seqlens_q[b] positions, so
 *     query i of b sits at position p = seq_lens_k[b] - nq_b + i and sees the
 *     causal context s = 0..p (n_t = p + 1 tokens, its own position included).
 *
 * Errors
 *   - Host-side checks (null pointers, alignment, unsupported sizes, a
 *     workspace that is too small) return DSA_ERR_INVALID_ARG,
 *     DSA_ERR_UNSUPPORTED or DSA_ERR_WORKSPACE and launch nothing.
 *   - A failed launch returns DSA_ERR_CUDA.
 *   - Device-side problems never trap: a bad length, page id or index is
 *     skipped (the affected row is left unspecified) and a bounded wait that
 *     runs out ends its block early; both set a device error word that
 *     dsa_check_device_error() reports (DSA_ERR_BAD_INDEX / DSA_ERR_TIMEOUT)
 *     and clears.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,  /* null pointer, misalignment, inconsistent sizes */
  DSA_ERR_UNSUPPORTED = 2,  /* sizes outside the supported set (see below) */
  DSA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  DSA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  DSA_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out */
  DSA_ERR_BAD_INDEX = 6,    /* a device-side length, page id or index was out of range */
  DSA_ERR_CAPACITY = 7      /* a device-side capacity was exceeded (HiSparse: rows of one step > slots) */
} dsa_status_t;

typedef enum { DSA_CACHE_CONTIGUOUS = 0, DSA_CACHE_PAGED = 1, DSA_CACHE_ROWS = 2 } dsa_cache_kind_t;

/*
 * A per-token row cache (indexer keys, or MLA latent rows) held in one pool of
 * rows.  Row r starts at  (bf16*)base + r * row_stride.
 *   contiguous: token s of sequence b is row seq_start[b] + s.
 *   paged:      token s of sequence b is row
 *                 page_table[b * page_table_stride + s / page_size] * page_size
 *                 + s % page_size.
 *   rows:       a position IS a pool row (no sequence addressing; sparse MLA
 *               only, e.g. over the HBM slots a HiSparse fetch returns).
 * Pages of a sequence beyond ceil(seq_lens_k[b] / page_size) are never read.
 */
typedef struct {
  int32_t kind;               /* dsa_cache_kind_t */
  int32_t page_size;          /* paged only: 64 */
  const void* base;           /* device, bf16 row pool */
  int64_t row_stride;         /* elements between rows (multiple of 8) */
  int64_t num_rows;           /* rows in the pool; a row id >= num_rows is a bad index */
  const int64_t* seq_start;   /* contiguous: device [num_seqs] */
  const int32_t* page_table;  /* paged: device [num_seqs, page_table_stride] */
  int64_t page_table_stride;  /* paged: entries per sequence */
} dsa_cache_t;

/* A ragged batch of query tokens. */
typedef struct {
  int32_t num_seqs;             /* B >= 1 */
  int32_t total_q;              /* T = cu_seqlens_q[B] (host copy, sizes the grids) */
  int32_t max_seqlen_k;         /* host upper bound of seq_lens_k[b] */
  int32_t max_q_per_seq;        /* host upper bound of cu_seqlens_q[b+1]-cu_seqlens_q[b] */
  const int32_t* cu_seqlens_q;  /* device [B+1], cu[0] = 0, non-decreasing */
  const int32_t* seq_lens_k;    /* device [B], nq_b <= seq_lens_k[b] <= max_seqlen_k */
} dsa_batch_t;

/* Lightning-indexer inputs.  Supported: n_heads in 1..64, head_dim in {32, 64, 128}. */
typedef struct {
  const void* q;       /* device bf16 [T, n_heads, head_dim], contiguous */
  const float* w;      /* device fp32 [T, n_heads], contiguous */
  dsa_cache_t k;       /* indexer keys: one head_dim bf16 row per token, shared by all heads */
  int32_t n_heads;
  int32_t head_dim;
} dsa_indexer_t;

/* One sparse-MLA layer.  Supported: n_heads in 1..64 and
 * (d_qk, d_v) in {(80, 64), (576, 512)}. */
typedef struct {
  const void* q;       /* device bf16 [T, n_heads, d_qk], contiguous */
  dsa_cache_t kv;      /* latent rows: d_qk bf16 per token; value = first d_v dims */
  int32_t n_heads;
  int32_t d_qk;
  int32_t d_v;
  float scale;         /* softmax scale applied to q . k */
} dsa_mla_layer_t;

/* Largest supported top-k and IndexShare group. */
#define DSA_MAX_TOPK 2048
#define DSA_MAX_LAYERS 4
/* Largest total_q of one call, and of total_q * n_layers for dsa_forward
 * (one grid row per query and layer); larger batches return
 * DSA_ERR_UNSUPPORTED: split them into several calls. */
#define DSA_MAX_QUERIES 65535

/* Human-readable name of a status code (static string, never NULL). */
const char* dsa_status_string(dsa_status_t status);

/*
 * Synchronises `stream`, then reads and clears the device error word set by
 * earlier kernels of this library on the current device.  Returns DSA_OK,
 * DSA_ERR_BAD_INDEX, DSA_ERR_TIMEOUT, DSA_ERR_CAPACITY, or DSA_ERR_CUDA if the
 * sync failed.
 */
dsa_status_t dsa_check_device_error(cudaStream_t stream);

/*
 * Bytes of device workspace the calls below need for `batch` and `topk`
 * (a per-query plan plus, for dsa_forward, the fp32 score matrix
 * [total_q, round_up(max_seqlen_k, 4)]).  0 on invalid arguments.
 */
size_t dsa_workspace_size(const dsa_batch_t* batch, int32_t topk);

/*
 * Step 1 alone: lightning-indexer scores.
 *   scores  device fp32 [total_q, ld_scores], ld_scores >= max_seqlen_k,
 *           multiple of 4.  Row t receives I[t, s] for s < n_t; entries
 *           s >= n_t are not written.
 *   skip_dense_k  queries with n_t <= skip_dense_k are skipped (their rows
 *           are not written; pass 0 to score every query, or the top-k to
 *           skip the rows dsa_topk takes whole).
 *   workspace  device, >= dsa_workspace_size(batch, 0) bytes.
 */
dsa_status_t dsa_indexer_scores(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                                int32_t skip_dense_k, float* scores, int64_t ld_scores,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Step 2 alone: exact top-k per query row of `scores` (layout as above; only
 * entries s < n_t are read).  Writes idx[t * ld_idx + j], j < topk: the
 * selected positions in ascending order, then -1 padding when n_t < topk.
 * topk in 1..2048.
 *   workspace  device, >= dsa_workspace_size(batch, 0) bytes (the per-call
 *              plan; the score matrix's share of that size is not used here).
 */
dsa_status_t dsa_topk(const dsa_batch_t* batch, const float* scores, int64_t ld_scores, int32_t topk,
                      int32_t* idx, int64_t ld_idx, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/*
 * Step 3 alone: sparse MLA over caller-supplied positions.
 *   idx    device int32 [total_q, ld_idx]; entry j < min(topk, n_t) of row t is
 *          a position of t's sequence, or -1 (skipped).  Entries at
 *          j >= min(topk, n_t) are never read.  A position outside [0, n_t)
 *          is skipped and flagged DSA_ERR_BAD_INDEX.  Repeated positions count
 *          as often as they appear.
 *   out    device bf16 [total_q, n_heads, d_v].
 *   lse    device fp32 [total_q, n_heads] (natural log of the softmax
 *          denominator, scale included), or NULL.  A row with no valid
 *          position gets out = 0 and lse = -inf.
 */
dsa_status_t dsa_sparse_mla_fwd(const dsa_batch_t* batch, const dsa_mla_layer_t* layer, const int32_t* idx,
                                int64_t ld_idx, int32_t topk, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * The fused forward: indexer (scores for the sparse queries only) -> top-k
 * (dense rows filled directly) -> sparse MLA for each of the n_layers layers
 * of an IndexShare group, all reading the one index set.
 *   idx    device int32 [total_q, ld_idx], written once (the cached top-k).
 *   outs   host array of n_layers device bf16 [total_q, n_heads, d_v] pointers.
 *   lses   host array of n_layers device fp32 [total_q, n_heads] pointers
 *          (entries may be NULL), or NULL.
 *          Output and LSE buffers may also be pinned (page-locked) host
 *          memory, which the device addresses directly: the results then land
 *          in host memory with no copy back (each is written once).
 *   workspace  device, >= dsa_workspace_size(batch, topk) bytes.
 */
dsa_status_t dsa_forward(const dsa_batch_t* batch, const dsa_indexer_t* indexer, int32_t topk,
                         int32_t n_layers, const dsa_mla_layer_t* layers, int32_t* idx, int64_t ld_idx,
                         void* const* outs, float* const* lses, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * The fused forward over compressed cache entries ("DeepSeek Sparse
 * Attention", In the code: the DeepSeek-V4 indexers score compressed KV
 * entries with ReLU(q.k) scores summed with weights and keep the top index_topk = 512 or
 * 1024 entries for compressed sparse attention).  Each cache row (indexer key
 * and latent row alike) is one entry standing for compress_ratio consecutive
 * tokens: entry j of sequence b covers tokens compress_ratio * j .. + ratio - 1
 * and takes row seq_start[b] + j (contiguous) or page_table[b, j / 64] * 64 +
 * j % 64 (paged, 64 entries a page).  seq_lens_k and max_seqlen_k still count
 * TOKENS, and the queries are the last tokens of each sequence; a query at
 * position p sees the (p + 1) / compress_ratio entries of complete blocks and
 * selects the topk of them (all of them when they are at most topk).  idx
 * holds entry indices.  Everything else as dsa_forward (`marks`: NULL, or five
 * timing events as in dsa_forward_marked); the same workspace size serves.
 * compress_ratio 1 is dsa_forward.
 */
dsa_status_t dsa_forward_compressed(const dsa_batch_t* batch, int32_t compress_ratio, const dsa_indexer_t* indexer,
                                    int32_t topk, int32_t n_layers, const dsa_mla_layer_t* layers, int32_t* idx,
                                    int64_t ld_idx, void* const* outs, float* const* lses, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream, cudaEvent_t const* marks);

/*
 * dsa_forward for a serving step whose inputs arrive while it runs: the
 * sparse-MLA launch waits for the caller's event `mla_ready` (recorded on
 * another stream once the layers' queries are uploaded and their latent rows
 * appended, so those copies overlap the indexer and the top-k), and
 * `topk_done` is recorded on `stream` once idx is written (the caller may copy
 * the index set back while the sparse MLA runs).  Either event may be NULL;
 * both NULL is dsa_forward.  Events are the caller's (cudaEventDefault or
 * cudaEventDisableTiming), and the call may be captured into a CUDA graph
 * with the other stream forked from `stream`.  Tokens only (no compressed
 * entries); everything else as dsa_forward.
 */
dsa_status_t dsa_forward_overlapped(const dsa_batch_t* batch, const dsa_indexer_t* indexer, int32_t topk,
                                    int32_t n_layers, const dsa_mla_layer_t* layers, int32_t* idx, int64_t ld_idx,
                                    void* const* outs, float* const* lses, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream, cudaEvent_t mla_ready, cudaEvent_t topk_done);

/*
 * dsa_forward with timing marks: identical work, plus cudaEventRecord of the
 * caller's events on `stream` -- marks[0] before the first launch, marks[1]
 * after the per-call plan, marks[2] after the indexer, marks[3] after the
 * top-k, marks[4] after the sparse-MLA launch.  `marks` holds 5 events
 * created by the caller (cudaEventDefault); NULL behaves like dsa_forward.
 */
dsa_status_t dsa_forward_marked(const dsa_batch_t* batch, const dsa_indexer_t* indexer, int32_t topk,
                                int32_t n_layers, const dsa_mla_layer_t* layers, int32_t* idx, int64_t ld_idx,
                                void* const* outs, float* const* lses, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream, cudaEvent_t const* marks);

/*
 * Cache append: the rows of a batch's query tokens into a row cache, so that
 * each new token is in its own causal context before the indexer scores it
 * (the top-k selector reads the whole context from HBM: "How GLM5.3 Sparse
 * Attention Affects HBM Memory Usage", What it claims / Model).  Call it once
 * for the indexer keys and once per layer for the latent rows.
 *   rows       device bf16 [total_q, ld_rows]: row t is query token t's new
 *              row (its first row_elems elements are copied).
 *   row_elems  multiple of 8, at most cache->row_stride; ld_rows >= row_elems,
 *              multiple of 8.
 *   cache      the pool is WRITTEN (through cache->base): query token t of
 *              sequence b at position p_t goes to the row that holds token
 *              p_t of b; no other row changes.  A page id out of range is
 *              skipped and flagged DSA_ERR_BAD_INDEX, and so is every token of a
 *              sequence whose lengths break the dsa_batch_t rules.
 * One launch, no workspace: each token's sequence is found on the device.
 * IndexShare: the index set dsa_forward writes is the group's stored top-k;
 * later layers of the group pass it to dsa_sparse_mla_fwd.
 */
dsa_status_t dsa_cache_append(const dsa_batch_t* batch, const void* rows, int64_t ld_rows, int32_t row_elems,
                              const dsa_cache_t* cache, cudaStream_t stream);

/*
 * HiSparse: HBM as a least-recently-used cache of one layer's latent rows over
 * host memory ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it
 * works / HiSparse (SGLang): rows chosen by top-k that are missing from HBM are
 * loaded from host DRAM, cold rows are evicted, the loads for layer N overlap
 * layer N-1).  The latent pool lives in host memory that the device can read
 * (pinned or registered host memory); `capacity` rows of it are held in a
 * device slot pool.  The cache is read-only: evicting a row drops it (host
 * memory keeps every row).  All buffers are caller-owned.
 */
typedef struct {
  int32_t capacity;     /* device slots (rows the HBM cache holds) */
  int32_t row_elems;    /* elements of a cached row (the latent width), multiple of 8 */
  void* slot_pool;      /* device bf16 [capacity, slot_stride] */
  int64_t slot_stride;  /* elements between slots, multiple of 8, >= row_elems */
  int64_t host_rows;    /* rows of the host pool (= the host cache's num_rows) */
  void* state;          /* device, >= dsa_hisparse_state_bytes(capacity, host_rows) bytes */
} dsa_hisparse_t;

/* Bytes of the device state of a cache (0 on invalid sizes). */
size_t dsa_hisparse_state_bytes(int32_t capacity, int64_t host_rows);

/* Workspace bytes of dsa_hisparse_fetch for this batch, top-k and capacity (0 on invalid arguments). */
size_t dsa_hisparse_workspace_size(const dsa_batch_t* batch, int32_t topk, int32_t capacity);

/* Empties the cache (every slot free, step counter 0).  Call once before the first fetch. */
dsa_status_t dsa_hisparse_reset(const dsa_hisparse_t* hs, cudaStream_t stream);

/*
 * One step: makes every row a batch selected resident and returns where.
 *   host_cache  the layer's latent cache in host memory: contiguous or paged
 *               addressing as for dsa_sparse_mla_fwd, base readable by the
 *               device, num_rows = hs->host_rows.
 *   idx         the selection, as for dsa_sparse_mla_fwd (entries j <
 *               min(topk, n_t); -1 entries skipped, bad ones flagged).
 *   slots       device int32 [total_q, ld_slots]: entry j of row t is the slot
 *               of idx[t, j]'s row, -1 where idx is -1 (and for j >= min(topk,
 *               n_t)).  Pass it to dsa_sparse_mla_fwd with a cache of kind
 *               DSA_CACHE_ROWS over slot_pool (num_rows = capacity).
 * Policy: the distinct requested rows in first-request order (row t, then
 * entry j); hits are resident, misses are copied from host memory into the
 * slots of the least recently used rows this step does not request; every
 * requested row becomes most recent (hits in their previous order, then the
 * misses in request order).  If the distinct rows of one step exceed
 * capacity, nothing changes, the error word reports DSA_ERR_CAPACITY and the
 * missing entries of `slots` are -1.
 * workspace: device, >= dsa_hisparse_workspace_size(batch, topk, capacity)
 * bytes, not shared with a call that may run at the same time (a fetch for
 * layer N on one stream beside layer N-1's attention on another needs its own).
 * Fetches of one cache run in stream order; a fetch and a sparse-MLA call
 * reading the same slots must be ordered by the caller (events or one stream).
 */
dsa_status_t dsa_hisparse_fetch(const dsa_hisparse_t* hs, const dsa_batch_t* batch, const dsa_cache_t* host_cache,
                                const int32_t* idx, int64_t ld_idx, int32_t topk, int32_t* slots, int64_t ld_slots,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The host rows held by the cache, least recently used first: rows[i] for the
 * i-th slot of the LRU order, -1 for a free slot.  rows: device int32 [capacity]. */
dsa_status_t dsa_hisparse_resident(const dsa_hisparse_t* hs, int32_t* rows, cudaStream_t stream);

/* Counters of the last fetch, copied to the host (synchronises `stream`):
 * stats[0] steps so far, [1] distinct rows requested, [2] hits, [3] misses
 * (rows loaded), [4] rows evicted, [5] 1 if the capacity was exceeded. */
dsa_status_t dsa_hisparse_stats(const dsa_hisparse_t* hs, int32_t* stats, cudaStream_t stream);

/*
 * MHA mode ("How GLM5.3 Sparse Attention Affects HBM Memory Usage", How it
 * works / Model: vLLM switches sparse MLA to MHA mode for contexts of about
 * 2K-5K tokens).  Instead of attending over the 576-dim latent rows with the
 * up-projections absorbed (MQA mode), every token of a short context is
 * up-projected once into per-head keys and values, and each head attends with
 * its own 256-dim query over the same top-k selection.  Shapes are fixed:
 * latent = 512 compressed dims + 64 rope dims (the latent row of the MQA
 * path), keys = 192 up-projected dims + the 64 rope dims, values = 256
 * up-projected dims.
 */
#define DSA_MHA_LATENT 512
#define DSA_MHA_ROPE 64
#define DSA_MHA_HEAD_DIM 256
#define DSA_MHA_MAX_HEADS 128
#define DSA_MHA_MAX_CONTEXT 131072

/*
 * dsa_mha_project -- per-head keys and values of `rows` latent rows:
 *   k_out[r, h, 0:192]   = W_UK[h] (192 x 512) . latent[r, 0:512]
 *   k_out[r, h, 192:256] = latent[r, 512:576]
 *   v_out[r, h, 0:256]   = W_UV[h] (256 x 512) . latent[r, 0:512]
 * latent: device bf16 [rows, latent_stride] (latent_stride >= 576, multiple
 * of 8); w_uk: device bf16 [n_heads, 192, 512]; w_uv: device bf16 [n_heads,
 * 256, 512]; k_out, v_out: device bf16 [rows, n_heads, 256] (written; rows
 * keep the latent pool's row numbers, so the latent cache's addressing serves
 * them).  bf16 operands, fp32 accumulation, bf16 results (round to nearest
 * even).  All pointers 16-byte aligned; rows <= 2^31 - 1; 1 <= n_heads <=
 * DSA_MHA_MAX_HEADS.  Asynchronous on `stream`.
 */
dsa_status_t dsa_mha_project(const void* latent, int64_t latent_stride, int64_t rows, int32_t n_heads,
                             const void* w_uk, const void* w_uv, void* k_out, void* v_out, cudaStream_t stream);

/* One MHA-mode attention layer. */
typedef struct {
  const void* q;        /* device bf16 [total_q, n_heads, 256]: per-head queries (192 no-rope + 64 rope dims) */
  dsa_cache_t k;        /* per-head keys: rows of n_heads x 256 bf16 (row_stride >= n_heads * 256),
                           addressed like the latent cache (contiguous or 64-token pages) */
  dsa_cache_t v;        /* per-head values, same row numbers and the same addressing as k */
  int32_t n_heads;      /* 1 .. DSA_MHA_MAX_HEADS */
  int32_t head_dim;     /* DSA_MHA_HEAD_DIM */
  int32_t v_head_dim;   /* DSA_MHA_HEAD_DIM */
  float scale;          /* softmax scale, > 0 (else DSA_ERR_INVALID_ARG), e.g. 1/sqrt(256) */
} dsa_mha_layer_t;

/* Workspace bytes of dsa_sparse_mha_fwd (the per-call plan and one selection
 * bit mask per query); 0 on invalid arguments. */
size_t dsa_mha_workspace_size(const dsa_batch_t* batch);

/*
 * dsa_sparse_mha_fwd -- for every query t and head h, softmax attention of
 * q[t, h] over the keys k[s, h] of the selected positions s (idx[t, j] for
 * j < min(topk, n_t); -1 entries skipped, out-of-range entries flagged
 * DSA_ERR_BAD_INDEX and skipped):
 *   z_s = scale * q[t, h] . k[s, h];  out[t, h] = sum_s softmax(z)_s v[s, h];
 *   lse[t, h] = log sum_s exp(z_s).
 * A query with no selected position gets out = 0 and lse = -inf.
 * out: device bf16 [total_q, n_heads, 256] (written); lse: device fp32
 * [total_q, n_heads] or NULL.  batch->max_seqlen_k <= DSA_MHA_MAX_CONTEXT.
 * bf16 operands, fp32 accumulation and softmax, probabilities rounded to bf16
 * for the value product.  workspace: >= dsa_mha_workspace_size(batch) bytes.
 */
dsa_status_t dsa_sparse_mha_fwd(const dsa_batch_t* batch, const dsa_mha_layer_t* layer, const int32_t* idx,
                                int64_t ld_idx, int32_t topk, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * dsa_sparse_mla_fwd_noalloc -- step 3 for callers that cannot provide any
 * device memory beyond their inputs and outputs (a plugin interface that
 * hands over only tensor pointers, or an engine whose device memory is all
 * claimed by its own pool, where a cudaMalloc at call time fails or stalls).
 * The pages describe no counterpart: this entry point exists for such callers.
 *
 * Same arguments, results and errors as dsa_sparse_mla_fwd, minus the
 * workspace: the per-call plan lives in a static device array of the library
 * (about 115 KB, held by every GPU that loads the library until exit).
 *   - total_q may be at most DSA_NOALLOC_MAX_QUERIES; larger batches return
 *     DSA_ERR_UNSUPPORTED without launching anything.
 *   - The first call on a device looks up that array's device address (one
 *     cudaGetSymbolAddress with the device current); make that first call
 *     before capturing a stream into a CUDA graph.
 *   - Nothing is allocated or freed, by the library or any library routine.
 *   - All calls share the one array, which keeps the last call's plan (each
 *     call rewrites every entry it reads).  Calls whose work overlaps on the
 *     GPU (different streams, or host threads) race on it: serialise them.
 */
#define DSA_NOALLOC_MAX_QUERIES 4096
dsa_status_t dsa_sparse_mla_fwd_noalloc(const dsa_batch_t* batch, const dsa_mla_layer_t* layer, const int32_t* idx,
                                        int64_t ld_idx, int32_t topk, void* out, float* lse, cudaStream_t stream);

/*
 * Self-checks of the library's own device machinery (test use).
 *
 * dsa_selftest_mma: one 128 x 64 tile D = A * B^T computed by the tensor-core
 * path the kernels use (bf16 operands staged in swizzled shared memory, fp32
 * accumulation in tensor memory).  A is bf16 [128, 64] row-major, B is bf16
 * [64, 64] row-major, D fp32 [128, 64].  `a_mn_major` / `b_mn_major` stage the
 * operand transposed (as the attention value and probability operands are).
 * `swizzle_bytes` is 128 (128-byte swizzled atoms of 64 K-elements) or 64
 * (64-byte swizzled atoms of 32 K-elements, K-major operands only, the way the
 * attention stages its rope halves), or 0: A is read from tensor memory (row m
 * in lane m, two elements per 32-bit column, the way MHA-mode attention feeds
 * its probabilities), B 128-byte swizzled; a_mn_major must be 0.
 *
 * dsa_selftest_topk_max_cluster: caps the thread-block cluster the top-k
 * launches use on the current device at `max_cluster` blocks (1, 2, 4, 8 or
 * 16; 0 restores the default), so tests can drive the paths taken when a row
 * is split over fewer blocks (long per-thread runs).  Host state only.
 *
 * dsa_selftest_topk_path: with `candidates` = 0 the top-k always takes its
 * three-pass path (every digit summed across the cluster, every block writes
 * its own selections); 1 (the default) lets it finish from the first digit's
 * candidates in one block when they fit.  Both give the same indices; tests
 * compare them.  Host state of the current device only.
 *
 * dsa_selftest_timeout: launches one block that waits on a barrier nobody
 * arrives at; the bounded wait gives up after about `limit_ms` milliseconds
 * and sets the device error word, which dsa_check_device_error then reports
 * as DSA_ERR_TIMEOUT.  Nothing faults; the context stays usable.
 */
dsa_status_t dsa_selftest_mma(const void* a, const void* b, float* d, int32_t a_mn_major, int32_t b_mn_major,
                              int32_t swizzle_bytes, cudaStream_t stream);
dsa_status_t dsa_selftest_topk_max_cluster(int32_t max_cluster);
dsa_status_t dsa_selftest_topk_path(int32_t candidates);
dsa_status_t dsa_selftest_timeout(int32_t limit_ms, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */

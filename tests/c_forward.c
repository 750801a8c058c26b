/* Plain-C client of the fused DSA forward: reads a problem written by the
 * test (contiguous caches, one layer), runs dsa_forward on device buffers
 * through the C ABI alone, and writes the indices, outputs and LSE back.
 *   usage: c_forward <input file> <output file>
 * Input: 11 int64 (B, T, max_seqlen_k, max_q_per_seq, H_I, d_I, H, D, D_v,
 * k, R pool rows), one float64 scale, then cu_seqlens_q int32 [B+1],
 * seq_lens_k int32 [B], q_idx bf16 [T,H_I,d_I], w fp32 [T,H_I], k_idx bf16
 * [R,d_I], q bf16 [T,H,D], kv bf16 [R,D], seq_start int64 [B].
 * Output: idx int32 [T,k], out bf16 [T,H,D_v], lse fp32 [T,H]. */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "dsa.h"

static int fail(const char* what) {
  fprintf(stderr, "c_forward: %s\n", what);
  return 1;
}

/* reads n bytes from f into a new device buffer */
static void* to_device(FILE* f, size_t n) {
  void* h = malloc(n ? n : 1);
  void* d = NULL;
  if (h == NULL || fread(h, 1, n, f) != n || cudaMalloc(&d, n ? n : 16) != cudaSuccess ||
      cudaMemcpy(d, h, n, cudaMemcpyHostToDevice) != cudaSuccess) {
    free(h);
    return NULL;
  }
  free(h);
  return d;
}

static int from_device(FILE* f, const void* d, size_t n) {
  void* h = malloc(n);
  int ok = h != NULL && cudaMemcpy(h, d, n, cudaMemcpyDeviceToHost) == cudaSuccess && fwrite(h, 1, n, f) == n;
  free(h);
  return ok;
}

int main(int argc, char** argv) {
  if (argc != 3) return fail("usage: c_forward <input> <output>");
  FILE* in = fopen(argv[1], "rb");
  if (in == NULL) return fail("cannot open the input");
  int64_t hd[11];
  double scale;
  if (fread(hd, sizeof(int64_t), 11, in) != 11 || fread(&scale, sizeof(double), 1, in) != 1)
    return fail("short header");
  const int64_t B = hd[0], T = hd[1], HI = hd[4], dI = hd[5], H = hd[6], D = hd[7], Dv = hd[8], k = hd[9],
                R = hd[10];
  void* cu = to_device(in, (size_t)(B + 1) * 4);
  void* lens = to_device(in, (size_t)B * 4);
  void* q_idx = to_device(in, (size_t)(T * HI * dI) * 2);
  void* w = to_device(in, (size_t)(T * HI) * 4);
  void* k_idx = to_device(in, (size_t)(R * dI) * 2);
  void* q = to_device(in, (size_t)(T * H * D) * 2);
  void* kv = to_device(in, (size_t)(R * D) * 2);
  void* seq_start = to_device(in, (size_t)B * 8);
  fclose(in);
  if (!cu || !lens || !q_idx || !w || !k_idx || !q || !kv || !seq_start) return fail("reading the inputs");

  dsa_batch_t batch = {(int32_t)B, (int32_t)T, (int32_t)hd[2], (int32_t)hd[3], (const int32_t*)cu,
                       (const int32_t*)lens};
  dsa_indexer_t ix;
  ix.q = q_idx;
  ix.w = (const float*)w;
  ix.k.kind = DSA_CACHE_CONTIGUOUS;
  ix.k.page_size = 0;
  ix.k.base = k_idx;
  ix.k.row_stride = dI;
  ix.k.num_rows = R;
  ix.k.seq_start = (const int64_t*)seq_start;
  ix.k.page_table = NULL;
  ix.k.page_table_stride = 0;
  ix.n_heads = (int32_t)HI;
  ix.head_dim = (int32_t)dI;
  dsa_mla_layer_t layer;
  layer.q = q;
  layer.kv = ix.k;
  layer.kv.base = kv;
  layer.kv.row_stride = D;
  layer.n_heads = (int32_t)H;
  layer.d_qk = (int32_t)D;
  layer.d_v = (int32_t)Dv;
  layer.scale = (float)scale;

  void *idx = NULL, *out = NULL, *lse = NULL, *ws = NULL;
  const size_t ws_bytes = dsa_workspace_size(&batch, (int32_t)k);
  if (ws_bytes == 0) return fail("dsa_workspace_size rejected the batch");
  if (cudaMalloc(&idx, (size_t)(T * k) * 4) != cudaSuccess || cudaMalloc(&out, (size_t)(T * H * Dv) * 2) != cudaSuccess ||
      cudaMalloc(&lse, (size_t)(T * H) * 4) != cudaSuccess || cudaMalloc(&ws, ws_bytes) != cudaSuccess)
    return fail("device allocation");
  void* outs[1] = {out};
  float* lses[1] = {(float*)lse};
  dsa_status_t s = dsa_forward(&batch, &ix, (int32_t)k, 1, &layer, (int32_t*)idx, k, outs, lses, ws, ws_bytes, NULL);
  if (s != DSA_OK) return fail(dsa_status_string(s));
  s = dsa_check_device_error(NULL);
  if (s != DSA_OK) return fail(dsa_status_string(s));

  FILE* o = fopen(argv[2], "wb");
  if (o == NULL) return fail("cannot open the output");
  if (!from_device(o, idx, (size_t)(T * k) * 4) || !from_device(o, out, (size_t)(T * H * Dv) * 2) ||
      !from_device(o, lse, (size_t)(T * H) * 4))
    return fail("writing the results");
  fclose(o);
  cudaFree(cu); cudaFree(lens); cudaFree(q_idx); cudaFree(w); cudaFree(k_idx); cudaFree(q); cudaFree(kv);
  cudaFree(seq_start); cudaFree(idx); cudaFree(out); cudaFree(lse); cudaFree(ws);
  printf("ok\n");
  return 0;
}

/* Plain-C client of libdsa.so: the header compiles as C99 and the host-side
 * entry points answer without a GPU (status strings, workspace sizing,
 * argument checks that return before any CUDA call).  Prints "ok" or the
 * first failed check and exits non-zero. */
#include <stdio.h>
#include <string.h>

#include "dsa.h"

#define CHECK(cond)                                    \
  do {                                                 \
    if (!(cond)) {                                     \
      printf("failed: %s (line %d)\n", #cond, __LINE__); \
      return 1;                                        \
    }                                                  \
  } while (0)

int main(void) {
  CHECK(strcmp(dsa_status_string(DSA_OK), "DSA_OK") == 0);
  CHECK(strncmp(dsa_status_string(DSA_ERR_WORKSPACE), "DSA_ERR_WORKSPACE", 17) == 0);
  CHECK(dsa_status_string((dsa_status_t)99) != NULL);

  /* a decode batch: 32 sequences of 32768 cached tokens, one query each (the
   * device pointers are never dereferenced by these calls) */
  static int32_t fake[64];
  dsa_batch_t b;
  b.num_seqs = 32;
  b.total_q = 32;
  b.max_seqlen_k = 32768;
  b.max_q_per_seq = 1;
  b.cu_seqlens_q = fake;
  b.seq_lens_k = fake;
  const size_t ws = dsa_workspace_size(&b, 2048);
  CHECK(ws >= (size_t)32 * 32768 * sizeof(float)); /* the fused call's score matrix */
  CHECK(dsa_workspace_size(NULL, 2048) == 0);
  CHECK(dsa_workspace_size(&b, 4096) == 0);          /* top-k above 2048 */

  /* argument checks that return before any CUDA call */
  CHECK(dsa_topk(&b, NULL, 32768, 2048, (int32_t*)fake, 2048, fake, ws, NULL) == DSA_ERR_INVALID_ARG);
  CHECK(dsa_topk(&b, (const float*)fake, 32768, 0, (int32_t*)fake, 2048, fake, ws, NULL) == DSA_ERR_UNSUPPORTED);
  CHECK(dsa_topk(&b, (const float*)fake, 32768, 2048, (int32_t*)fake, 2048, fake, 16, NULL) == DSA_ERR_WORKSPACE);
  CHECK(dsa_cache_append(&b, fake, 576, 576, NULL, NULL) == DSA_ERR_INVALID_ARG);
  b.num_seqs = 0;
  CHECK(dsa_workspace_size(&b, 2048) == 0);           /* no sequences */
  printf("ok\n");
  return 0;
}

/* A plain C99 program against the C ABI: the header compiles as C, the library
 * links and loads without C++ or PyTorch, and calls that fail host validation
 * return their status without touching a GPU. */
#include <stdio.h>
#include <string.h>

#include "triforce_attn.h"

static int failures = 0;

static void expect(int got, int want, const char* what) {
  if (got != want) {
    printf("FAIL %s: got %d, want %d\n", what, got, want);
    ++failures;
  }
}

int main(void) {
  uint16_t* fake = (uint16_t*)(uintptr_t)0x10000; /* never dereferenced */
  int32_t* ifake = (int32_t*)(uintptr_t)0x10000;
  float* ffake = (float*)(uintptr_t)0x10000;

  expect(tf_abi_version() / 100, 1, "ABI major version");
  expect(strcmp(tf_status_string(TF_OK), "ok"), 0, "status string of TF_OK");
  expect(tf_status_string(TF_ERR_DEVICE_DATA)[0] != '\0', 1, "status string of TF_ERR_DEVICE_DATA");

  expect(tf_build_chunk_means(NULL, ifake, 1, 1, 64, 128, 8, 0, 8, fake, NULL), TF_ERR_INVALID_ARG,
         "chunk means without K");
  expect(tf_build_chunk_means(fake, ifake, 1, 1, 64, 64, 8, 0, 8, fake, NULL), TF_ERR_UNSUPPORTED,
         "chunk means with D = 64");
  expect(tf_sparse_decode_attn(fake, fake, fake, ifake, ifake, ifake, 1, 8, 2, 64, 128, 8, 4, 0.1f, ffake, NULL, 0,
                               NULL),
         TF_ERR_WORKSPACE, "sparse decode without workspace");
  expect(tf_pack_retrieval_cache(fake, fake, ifake, ifake, ifake, 1, 2, 64, 128, 8, 4097, fake, fake, ifake, ifake,
                                 NULL),
         TF_ERR_UNSUPPORTED, "packing with kc above 4096");
  expect(tf_retrieval_window_draft_attn(fake, fake, fake, fake, ifake, 1, 8, 2, 64, 128, 8, 4, 0.1f, NULL, 4, 60,
                                        ifake, ifake, NULL, ffake, NULL, NULL),
         TF_ERR_INVALID_ARG, "window draft without a window output");
  expect(tf_retrieval_window_draft_attn(fake, fake, fake, fake, ifake, 1, 2, 2, 64, 128, 8, 4, 0.1f, NULL, 4, 60,
                                        ifake, ifake, NULL, ffake, ffake, NULL),
         TF_ERR_UNSUPPORTED, "window draft with one query head per KV head");
  expect(tf_check_status(NULL, 4096, NULL), TF_ERR_INVALID_ARG, "status of a missing workspace");
  expect(tf_chunk_scores_topk_workspace(1, 32, 131072, 8) == 0, 1, "top-k needs no workspace");

  if (failures == 0) printf("c consumer ok\n");
  return failures == 0 ? 0 : 1;
}

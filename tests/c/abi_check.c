/* Host-only use of the C ABI from plain C99: the header compiles as C, the
 * library links, and argument validation answers before any launch. */
#include <stdio.h>
#include <string.h>

#include "attn.h"

static int fails = 0;

static void expect(int cond, const char* what) {
  if (!cond) {
    printf("FAIL %s\n", what);
    ++fails;
  }
}

int main(void) {
  void* fake = (void*)(size_t)0x10000; /* 16-byte aligned, never dereferenced */
  expect(strcmp(attn_status_string(ATTN_OK), "ATTN_OK") == 0, "status string");
  expect(attn_fwd(NULL, fake, fake, fake, (float*)fake, 1, 128, 128, 2, 2, 64, 0.125f, 0, NULL, ATTN_BF16, NULL) ==
             ATTN_ERR_INVALID_ARG,
         "null q");
  expect(strlen(attn_last_error()) > 0, "last error text");
  expect(attn_fwd(fake, fake, fake, fake, (float*)fake, 1, 128, 128, 2, 2, 96, 0.125f, 0, NULL, ATTN_BF16, NULL) ==
             ATTN_ERR_UNSUPPORTED,
         "head_dim 96");
  expect(attn_bwd_workspace_size(2, 300, 4, 128, 1, ATTN_BF16) > 0, "workspace size");
  expect(attn_bwd(fake, fake, fake, fake, (const float*)fake, fake, fake, fake, fake, 2, 300, 300, 4, 4, 128, 0.1f, 0,
                  NULL, ATTN_BF16, 1, fake, 16, NULL) == ATTN_ERR_WORKSPACE,
         "small workspace");
  expect(attn_segment_info_size(2, 300, 129) == 2 * (3 + 2) * 16, "segment info size");
  expect(attn_decode_num_splits(8, 1, 131072, 32, 8, 128) >= 1, "decode splits");
  expect(attn_fwd_num_splits(4, 2048, 16384, 8, 128, 1, ATTN_BF16) == 2, "forward splits");
  expect(attn_fwd_split(fake, fake, fake, fake, (float*)fake, 2, 300, 4096, 4, 2, 64, 0.125f, -1, 0, NULL, 3, NULL,
                        0, ATTN_BF16, NULL) == ATTN_ERR_WORKSPACE,
         "split forward without workspace");
  printf("%s\n", fails ? "FAILED" : "OK");
  return fails ? 1 : 0;
}

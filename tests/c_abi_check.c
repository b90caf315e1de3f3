/* Compiled and run by tests/test_host.py: include/dsa.h is plain C, and a C
 * program links libdsa.so and gets the documented host-side answers without
 * touching a GPU. */
#include <stdio.h>
#include <string.h>

#include "dsa.h"

int main(void) {
  if (strstr(dsa_version(), "sm_103a") == NULL) return 2;
  /* host-side validation: a null pointer is rejected before any launch */
  if (dsa_topk(NULL, 100, NULL, NULL, 1, 1, 10, NULL, NULL, 0, NULL) != DSA_ERR_INVALID_ARG) return 3;
  if (strstr(dsa_last_error(), "null") == NULL) return 4;
  /* nothing to do succeeds */
  if (dsa_topk(NULL, 100, NULL, NULL, 1, 0, 10, NULL, NULL, 0, NULL) != DSA_OK) return 5;
  /* split partials: T*H*S*(4*Dv + 8) bytes */
  if (sparse_mla_workspace_size(8, 128, 512, 8) != (size_t)8 * 128 * 8 * (512 * 4 + 8)) return 6;
  if (dsa_topk_workspace_size(32, 8192, 2048) != 0) return 7;
  printf("c abi ok\n");
  return 0;
}

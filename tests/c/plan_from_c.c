/* Plans through the C ABI from plain C99 (no CUDA call, no framework):
 * pkd_abi_version, pkd_workspace_size, pkd_plan_host and
 * pkd_plan_shared_prefix_host, then prints the plan fields and the image
 * words so that a test can compare them with the Python binding's plans.
 * Usage: plan_from_c  (fixed small problem, output on stdout) */
#include <stdio.h>
#include <stdlib.h>

#include "pkd.h"

int main(void) {
  if (pkd_abi_version() != PKD_ABI_VERSION) {
    fprintf(stderr, "ABI version %d, header %d\n", pkd_abi_version(), PKD_ABI_VERSION);
    return 1;
  }
  pkd_problem p = {0};
  p.batch = 3;
  p.num_qo_heads = 32;
  p.num_kv_heads = 8;
  p.head_dim = 128;
  p.page_size = 16;
  p.dtype = PKD_F16;
  p.num_pages = 64;
  p.num_ctas = 7;
  p.min_chunks_per_request = 2;
  /* three requests: 5 pages (last holds 9 tokens), none, 2 pages (full) */
  const int32_t indptr[4] = {0, 5, 5, 7};
  const int32_t last[3] = {9, 1, 16};
  const int32_t indices[7] = {3, 17, 40, 2, 63, 11, 12};
  size_t int_ws = 0, float_ws = 0, staging = 0;
  if (pkd_workspace_size(&p, &int_ws, &float_ws, &staging) != PKD_OK) {
    fprintf(stderr, "workspace_size: %s\n", pkd_last_error());
    return 1;
  }
  int32_t *image = (int32_t *)calloc(int_ws / 4 + 1, sizeof(int32_t));
  pkd_plan_t plan;
  if (pkd_plan_host(&p, indptr, last, indices, &plan, image, int_ws) != PKD_OK) {
    fprintf(stderr, "plan_host: %s\n", pkd_last_error());
    return 1;
  }
  printf("plan %d %d %d %lld %lld\n", plan.num_units, plan.num_partials,
         plan.num_split_requests, (long long)plan.total_tokens,
         (long long)plan.int_ws_bytes_used);
  printf("image");
  for (long long i = 0; i < plan.int_ws_bytes_used / 4; ++i) printf(" %d", image[i]);
  printf("\n");
  /* a page id outside the pool is refused with PKD_ERR_PAGE_TABLE */
  const int32_t bad[7] = {3, 17, 64, 2, 63, 11, 12};
  pkd_status st = pkd_plan_host(&p, indptr, last, bad, &plan, image, int_ws);
  printf("bad_page %d\n", (int)st);
  /* shared prefix: 3 pages, last holds 5 tokens */
  pkd_problem q = p;
  q.num_ctas = 16;
  q.min_chunks_per_request = 1;
  const int32_t prefix[3] = {4, 9, 2};
  int32_t pimage[32] = {0};
  pkd_prefix_plan_t pplan;
  if (pkd_plan_shared_prefix_host(&q, prefix, 3, 5, &pplan, pimage, sizeof(pimage)) != PKD_OK) {
    fprintf(stderr, "plan_shared_prefix_host: %s\n", pkd_last_error());
    return 1;
  }
  printf("prefix %d %d %d %d\n", pplan.prefix_len, pplan.chunks, pplan.chunk_tiles,
         pplan.row_tiles);
  printf("pimage");
  for (long long i = 0; i < pplan.int_ws_bytes_used / 4; ++i) printf(" %d", pimage[i]);
  printf("\n");
  free(image);
  return 0;
}

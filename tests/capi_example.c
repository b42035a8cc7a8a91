/* A C program using the library through include/cp_api.h alone: the host-side
 * helpers (chunk plan, query-width ladder, rolling alignment, token-budget
 * schedule, workspace size), which need no GPU.  tests/test_capi_c.py builds
 * it with gcc against libcp.so and checks what it prints. */
#include <stdio.h>

#include "cp_api.h"

int main(void) {
  int32_t sizes[16];
  const int32_t n = cp_chunk_plan(4000, 512, sizes, 16);
  printf("abi %d\nplan %d:", (int)cp_abi_version(), (int)n);
  for (int i = 0; i < n && i < 16; ++i) printf(" %d", (int)sizes[i]);
  int32_t tiers[3];
  const int32_t nt = cp_query_ladder(512, tiers);
  printf("\nladder %d:", (int)nt);
  for (int i = 0; i < nt; ++i) printf(" %d", (int)tiers[i]);
  printf("\nwidth416 %d\naligned %d\n", (int)cp_query_width(416, 512), (int)cp_aligned_length(2000, 256));
  const int32_t prompts[4] = {20000, 20000, 20000, 20000};
  static cp_sched_entry plan[4096];
  const int32_t ne = cp_schedule(8192, 64, prompts, 4, plan, 4096);
  int steps = 0, rows0 = 0;
  for (int i = 0; i < ne && i < 4096; ++i) {
    if (plan[i].step + 1 > steps) steps = plan[i].step + 1;
    if (plan[i].step == 0) rows0 += plan[i].rows;
  }
  printf("schedule %d entries, %d steps, step 0 rows %d\n", (int)ne, steps, rows0);
  cp_layer_desc d = {CP_BF16, 1, 32, 8, 128, CP_CACHE_CONTIG, 8192, 0, 0, 0, 0.f};
  printf("workspace %zu\n", cp_workspace_size(&d, 512, 8192, 1));
  printf("rows past the chunk: %s\n", cp_status_string(cp_query_width(600, 512)));
  return 0;
}

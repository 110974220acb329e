/*
 * Plans one MSA prefill layout through the C ABI of libmsa.so from plain C99 (host-only
 * entry points: no GPU call), and prints what the test compares.
 *
 * Layout: one sequence; pool blocks 1 and 0 hold positions 0-15 and 16-31 (one segment of
 * two logical blocks); the chunk holds positions 32..40.  Hq = 4, Hkv = 2, d = 64.
 */
#include <stdio.h>
#include <stdlib.h>

#include "msa.h"

static msa_plan_opts_t opts(void) {
  msa_plan_opts_t o = {0};
  o.num_heads_q = 4;
  o.num_heads_kv = 2;
  o.head_dim = 64;
  o.block_size = 16;
  return o;
}

int main(void) {
  const msa_plan_opts_t o = opts();
  const msa_segment_t seg = {0, 0, 2};
  const int32_t block_table[2] = {1, 0};
  const int32_t block_pos[2] = {16, 0};
  const int32_t block_fill[2] = {16, 16};
  const int32_t cu_q[2] = {0, 9};
  int32_t q_pos[9];
  for (int i = 0; i < 9; ++i) q_pos[i] = 32 + i;

  msa_plan_t* plan = NULL;
  msa_status_t st = msa_plan_create(&o, MSA_PREFILL, 1, &seg, 1, block_table, 2, block_pos, block_fill, 2,
                                    cu_q, q_pos, &plan);
  if (st != MSA_OK || plan == NULL) {
    printf("create failed: %d %s\n", (int)st, msa_status_string(st));
    return 1;
  }
  msa_plan_stats_t s;
  if (msa_plan_get_stats(plan, &s) != MSA_OK) return 1;
  size_t n = 0;
  if (msa_plan_export(plan, NULL, 0, &n) != MSA_OK || n == 0) return 1;
  int32_t* ex = (int32_t*)malloc(n * sizeof(int32_t));
  if (!ex || msa_plan_export(plan, ex, n, &n) != MSA_OK) return 1;

  printf("version %d\n", (int)msa_version());
  printf("useful_flops %lld\n", (long long)s.useful_flops);
  printf("kv_tokens %lld\n", (long long)s.kv_tokens);
  printf("export");
  for (size_t i = 0; i < n; ++i) printf(" %d", (int)ex[i]);
  printf("\n");
  free(ex);
  msa_plan_destroy(plan);

  /* a chunk position that a pool block already holds is refused and leaves the plan NULL */
  q_pos[0] = 31;
  plan = (msa_plan_t*)&st; /* any non-NULL value: the call must reset it */
  st = msa_plan_create(&o, MSA_PREFILL, 1, &seg, 1, block_table, 2, block_pos, block_fill, 2, cu_q, q_pos, &plan);
  printf("overlap %d %s\n", (int)st, plan == NULL ? "null" : "set");
  return 0;
}

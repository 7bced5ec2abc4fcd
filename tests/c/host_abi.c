/* The library's host entry points used from plain C (no Python, no CUDA
 * calls): a block allocator scenario with a fork and a copy-on-write append,
 * the chunked-prefill step planner, and the split-K partition chooser and
 * work order.  Prints "ok" and exits 0 when every check holds. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "pa.h"

#define CHECK(c)                                                   \
  do {                                                             \
    if (!(c)) {                                                    \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
      return 1;                                                    \
    }                                                              \
  } while (0)

int main(void) {
  /* 8 blocks of 16 tokens, free list 0, 1, ..., 7 */
  pa_alloc* a = NULL;
  CHECK(pa_alloc_create(8, 16, NULL, &a) == PA_OK && a != NULL);
  CHECK(pa_alloc_add_seq(a, 7) == PA_OK);
  int32_t src = 0, dst = 0;
  CHECK(pa_alloc_reserve(a, 7, 20, &src, &dst) == PA_OK);  /* blocks 0, 1 */
  CHECK(src == -1 && dst == -1);
  int32_t table[4];
  int n = 0;
  CHECK(pa_alloc_block_table(a, 7, table, 4, &n) == PA_OK && n == 2);
  CHECK(table[0] == 0 && table[1] == 1);
  CHECK(pa_alloc_tail_waste(a, 7) == 12);                  /* 32 slots, 20 used */
  /* fork: the child shares both blocks; its next token lands in the shared,
   * partly filled block 1, so it moves to a fresh block (2) first */
  CHECK(pa_alloc_fork(a, 7, 9) == PA_OK);
  CHECK(pa_alloc_refcount(a, 0) == 2 && pa_alloc_refcount(a, 1) == 2);
  int64_t slot = -1;
  CHECK(pa_alloc_append_slot(a, 9, &slot, &src, &dst) == PA_OK);
  CHECK(src == 1 && dst == 2);
  CHECK(slot == 2 * 16 + 4);                               /* position 20 of block 2 */
  CHECK(pa_alloc_refcount(a, 1) == 1 && pa_alloc_refcount(a, 2) == 1);
  /* the parent's own next token stays in its block 1 */
  CHECK(pa_alloc_append_slot(a, 7, &slot, &src, &dst) == PA_OK);
  CHECK(slot == 1 * 16 + 4 && src == -1 && dst == -1);
  CHECK(pa_alloc_num_free(a) == 5);
  CHECK(pa_alloc_free_seq(a, 9) == PA_OK);
  CHECK(pa_alloc_refcount(a, 0) == 1 && pa_alloc_num_free(a) == 6);
  pa_alloc_destroy(a);

  /* step planner: budget 2048, 60 decodes, a 10,000-token prompt */
  int32_t remaining = 10000, chunk = 0;
  int decodes = 0;
  CHECK(pa_plan_step(2048, 60, &remaining, 1, &chunk, &decodes) == PA_OK);
  CHECK(decodes == 60 && chunk == 1988);

  /* partition chooser and work order */
  const int32_t ctx[4] = {100, 3000, 17, 1500};
  const int part = pa_splitk_partition_size(ctx, 4, 32, 8, 128, 0, 152, 1);
  CHECK(part >= 256 && part % 16 == 0);
  int32_t order[2 * 4];
  CHECK(pa_splitk_order(ctx, 4, 1536, 2, order) == 8);
  /* items: part * 4 + b; tokens 100, 1536, 17, 1500 | 0, 1464, 0, 0 */
  CHECK(order[0] == 1 && order[1] == 3 && order[2] == 5 && order[3] == 0 && order[4] == 2);
  CHECK(pa_splitk_order(ctx, 4, 0, 2, order) == -1);

  printf("ok\n");
  return 0;
}

/* The host block pool through the C ABI alone, from plain C (no Python):
 * the OS-lab appendix's copy-on-write walk-through at block size 4 (section
 * 4.4: after a fork both sequences share every block; the first writer into
 * the shared partial block gets a copy, the last holder writes in place),
 * refcounts through free, and the error statuses, the batched token append's
 * short count among them.  Exit status 0 when every
 * check holds; the first failing check is printed. */
#include <stdint.h>
#include <stdio.h>

#include "pagedattn.h"

static int failures = 0;
#define CHECK(cond)                                                   \
  do {                                                                \
    if (!(cond)) {                                                    \
      printf("check failed at line %d: %s (%s)\n", __LINE__, #cond,   \
             pa_last_error() ? pa_last_error() : "");                 \
      ++failures;                                                     \
      return 1;                                                       \
    }                                                                 \
  } while (0)

static int rc_of(pa_pool* pool, int block) {
  int rc = -1;
  if (pa_pool_refcount(pool, block, &rc) != PA_OK) return -1;
  return rc;
}

static int cow_walkthrough(void) {
  pa_pool* pool = NULL;
  CHECK(pa_pool_create(8, 4, NULL, &pool) == PA_OK && pool);
  int a = -1, b = -1;
  CHECK(pa_pool_new_seq(pool, &a) == PA_OK);
  int64_t slot, src, dst;
  for (int t = 0; t < 6; ++t) {  /* 6 tokens: one full block, one holding 2 */
    CHECK(pa_pool_append_slot(pool, a, &slot, &src, &dst) == PA_OK);
    CHECK(src == -1 && dst == -1);  /* nothing shared yet */
  }
  int32_t ta[4];
  int n = 0, ctx = 0;
  CHECK(pa_pool_block_table(pool, a, ta, 4, &n, &ctx) == PA_OK && n == 2 && ctx == 6);
  CHECK(pa_pool_fork(pool, a, &b) == PA_OK && b != a);
  CHECK(rc_of(pool, ta[0]) == 2 && rc_of(pool, ta[1]) == 2);  /* the table, not the data */

  /* a writes into the shared partial block: it gets a copy first */
  CHECK(pa_pool_append_slot(pool, a, &slot, &src, &dst) == PA_OK);
  CHECK(src == ta[1] && dst >= 0 && dst != ta[1]);
  CHECK(slot == dst * 4 + 2);  /* offset 2 of the copy */
  CHECK(rc_of(pool, ta[1]) == 1 && rc_of(pool, (int)dst) == 1);

  /* b is now the last holder of the old block: it writes in place */
  CHECK(pa_pool_append_slot(pool, b, &slot, &src, &dst) == PA_OK);
  CHECK(src == -1 && dst == -1 && slot == (int64_t)ta[1] * 4 + 2);

  pa_pool_stats_t st;
  CHECK(pa_pool_stats(pool, &st) == PA_OK && st.cow_copies == 1 && st.live_seqs == 2);
  CHECK(st.shared_blocks == 1);  /* block 0 */

  CHECK(pa_pool_free_seq(pool, a) == PA_OK);
  CHECK(rc_of(pool, ta[0]) == 1);
  CHECK(pa_pool_free_seq(pool, b) == PA_OK);
  CHECK(pa_pool_stats(pool, &st) == PA_OK && st.free_blocks == 8 && st.used_blocks == 0);
  CHECK(pa_pool_destroy(pool) == PA_OK);
  return 0;
}

static int errors(void) {
  pa_pool* pool = NULL;
  CHECK(pa_pool_create(1, 4, NULL, &pool) == PA_OK);
  int s = -1, child = -1;
  int64_t slot, src, dst;
  CHECK(pa_pool_fork(pool, 12345, &child) == PA_ERR_NOT_FOUND);
  CHECK(pa_pool_new_seq(pool, &s) == PA_OK);
  for (int t = 0; t < 4; ++t) CHECK(pa_pool_append_slot(pool, s, &slot, &src, &dst) == PA_OK);
  /* the fifth token needs a second block: refused, the pool unchanged */
  CHECK(pa_pool_append_slot(pool, s, &slot, &src, &dst) == PA_ERR_NO_BLOCKS);
  int n = 0, ctx = 0;
  CHECK(pa_pool_block_table(pool, s, NULL, 0, &n, &ctx) == PA_OK && n == 1 && ctx == 4);
  CHECK(pa_pool_free_seq(pool, s) == PA_OK);
  CHECK(pa_pool_free_seq(pool, s) == PA_ERR_NOT_FOUND);  /* no double free */
  CHECK(pa_pool_destroy(pool) == PA_OK);
  CHECK(pa_pool_create(4, 0, NULL, &pool) == PA_ERR_INVALID_ARG);

  /* the batched token append: 6 tokens into a 1-block pool stop after 4 */
  CHECK(pa_pool_create(1, 4, NULL, &pool) == PA_OK);
  CHECK(pa_pool_new_seq(pool, &s) == PA_OK);
  int32_t seqs[6], toks[6];
  int64_t slots[6], pairs[12];
  for (int t = 0; t < 6; ++t) { seqs[t] = s; toks[t] = 7 + t; }
  int np = -1, done = -1;
  CHECK(pa_pool_append_tokens(pool, seqs, toks, 6, slots, NULL, 6, &np, &done) ==
        PA_ERR_INVALID_ARG);  /* pairs NULL with room claimed */
  CHECK(pa_pool_append_tokens(pool, seqs, toks, 6, slots, pairs, 6, &np, &done) ==
        PA_ERR_NO_BLOCKS);
  CHECK(done == 4 && np == 0 && slots[0] == 0 && slots[3] == 3);
  CHECK(pa_pool_append_tokens(pool, seqs, toks, 0, NULL, NULL, 0, &np, &done) == PA_OK &&
        done == 0);
  CHECK(pa_pool_destroy(pool) == PA_OK);

  /* a copy pair with no room for it: refused before that append, the ones
   * before it kept */
  CHECK(pa_pool_create(4, 4, NULL, &pool) == PA_OK);
  CHECK(pa_pool_new_seq(pool, &s) == PA_OK);
  seqs[0] = seqs[1] = s;
  CHECK(pa_pool_append_tokens(pool, seqs, toks, 2, slots, pairs, 0, &np, &done) == PA_OK &&
        done == 2);
  CHECK(pa_pool_fork(pool, s, &child) == PA_OK);
  int32_t two[2] = {child, s};
  CHECK(pa_pool_append_tokens(pool, two, toks, 2, slots, NULL, 0, &np, &done) ==
        PA_ERR_INVALID_ARG);
  CHECK(done == 0 && np == 0);
  CHECK(pa_pool_append_tokens(pool, two, toks, 2, slots, pairs, 1, &np, &done) == PA_OK);
  CHECK(done == 2 && np == 1);  /* the child copies; the parent then writes in place */
  CHECK(pa_pool_destroy(pool) == PA_OK);
  return 0;
}

int main(void) {
  cow_walkthrough();
  errors();
  if (failures == 0) printf("pool C ABI: all checks passed\n");
  return failures == 0 ? 0 : 1;
}

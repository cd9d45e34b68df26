/* The C ABI used from C: this file is compiled as C11 against include/gdn.h
 * and linked to libgdn.so by tests/test_c_abi.py. It calls only what needs no
 * GPU: version and error strings, argument validation that happens before
 * any device work, the rollback table, slot addresses and the checkpoint
 * selector. Exit status 0 = every check held. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gdn.h"

static int failures = 0;
#define CHECK(cond)                                                      \
  do {                                                                   \
    if (!(cond)) {                                                       \
      fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
      ++failures;                                                        \
    }                                                                    \
  } while (0)

int main(void) {
  CHECK(strstr(gdn_version(), "sm_103a") != NULL);

  /* validation before any device work */
  CHECK(gdn_forward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, GDN_MODE_GDA,
                    NULL) == GDN_ERR_INVALID_ARG);
  CHECK(strlen(gdn_last_error()) > 0);
  gdn_shape sh;
  memset(&sh, 0, sizeof sh);
  sh.n_seqs = 2; sh.T = 3; sh.H = 2; sh.D_k = 32; sh.D_v = 128; sh.in_dtype = GDN_BF16;
  float fake_f[4];
  const void *fake = (const void *)((size_t)1 << 20); /* aligned, never dereferenced */
  CHECK(gdn_forward(&sh, fake, fake, fake, (const float *)fake, (const float *)fake,
                    (const float *const *)fake, (float *)fake, (float *)fake, 1, GDN_MODE_GDA,
                    NULL) == GDN_ERR_UNSUPPORTED);
  sh.D_k = 128;
  CHECK(gdn_forward(&sh, fake, fake, fake, (const float *)fake, (const float *)fake,
                    (const float *const *)fake, (float *)fake, (float *)fake, 0, GDN_MODE_GDA,
                    NULL) == GDN_ERR_INVALID_ARG); /* n_slots = 0 */
  sh.n_seqs = 0; /* nothing to do: no device needed */
  CHECK(gdn_forward(&sh, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, GDN_MODE_GDA,
                    NULL) == GDN_OK);
  (void)fake_f;

  gdn_varlen_shape vs;
  memset(&vs, 0, sizeof vs);
  vs.n_seqs = 2; vs.total_tokens = 100; vs.H = 2; vs.D_k = 128; vs.D_v = 128;
  vs.in_dtype = GDN_BF16;
  CHECK(gdn_chunked_workspace_size(&vs, 8) > 0);
  CHECK(gdn_chunked_workspace_size(&vs, 0) == 0);
  CHECK(gdn_noalloc_scratch_bytes() == ((size_t)256 << 20));

  /* rollback table: T = 8 tokens, K = 3 slots */
  gdn_seq_table *t = NULL;
  CHECK(gdn_seq_table_create(4, 3, &t) == GDN_OK && t != NULL);
  CHECK(gdn_seq_table_record(t, 1, 8) == GDN_OK);
  int slot = 99;
  CHECK(gdn_rollback(t, 1, 0, &slot) == GDN_OK && slot == -1);
  CHECK(gdn_rollback(t, 1, 8, &slot) == GDN_OK && slot == 2);
  CHECK(gdn_rollback(t, 1, 6, &slot) == GDN_OK && slot == 0);
  CHECK(gdn_rollback(t, 1, 5, &slot) == GDN_ERR_ROLLBACK_RANGE);
  CHECK(gdn_rollback(t, 1, 9, &slot) == GDN_ERR_ROLLBACK_RANGE);
  CHECK(gdn_seq_table_record(t, 7, 1) == GDN_ERR_INVALID_ARG);
  CHECK(gdn_seq_table_clear(t, 1) == GDN_OK);
  CHECK(gdn_rollback(t, 1, 0, &slot) == GDN_OK && slot == -1);
  gdn_seq_table_destroy(t);

  /* slot addresses: fp32 [N][K][H][D_k][D_v] */
  const float *base = (const float *)((size_t)1 << 30), *p = NULL;
  CHECK(gdn_slot_state_ptr(base, 2, 1, 3, 4, 64, 64, &p) == GDN_OK);
  CHECK(p == base + ((2 * 3 + 1) * 4) * 64 * 64);
  CHECK(gdn_slot_state_ptr(base, 0, -1, 3, 4, 64, 64, &p) == GDN_OK && p == NULL);

  /* checkpoint selector: L = 300, 4 slots, a checkpoint every 64, at most 3 */
  int src = -1, idx = -1, rep = -1;
  CHECK(gdn_checkpoint_select(298, 300, 4, 64, 3, &src, &idx, &rep) == GDN_OK);
  CHECK(src == 2 && idx == 1 && rep == 298);     /* slot 1 holds 298 tokens */
  CHECK(gdn_checkpoint_select(250, 300, 4, 64, 3, &src, &idx, &rep) == GDN_OK);
  CHECK(src == 1 && idx == 2 && rep == 192);     /* last checkpoint: 3 x 64 */
  CHECK(gdn_checkpoint_select(63, 300, 4, 64, 3, &src, &idx, &rep) == GDN_OK);
  CHECK(src == 0 && idx == -1 && rep == 0);
  CHECK(gdn_checkpoint_select(301, 300, 4, 64, 3, &src, &idx, &rep) == GDN_ERR_INVALID_ARG);
  CHECK(gdn_checkpoint_select(10, 300, 4, 96, 3, &src, &idx, &rep) == GDN_ERR_INVALID_ARG);

  if (failures) fprintf(stderr, "%d check(s) failed\n", failures);
  else printf("c abi host checks passed\n");
  return failures ? 1 : 0;
}

/* A plain C99 client of liblce.so: the headers compile as C, the library
 * links and loads without Python or torch, and the host-side contract holds
 * without a GPU (workspace queries, argument checks that launch nothing,
 * status strings, kernel accounting names). Prints "C-ABI-OK" on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "lce.h"
#include "lce_testing.h"

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
      return 1;                                                  \
    }                                                            \
  } while (0)

int main(void) {
  /* workspace size: positive, grows with N, the chunk hint bounds it */
  size_t a = lce_workspace_size(LCE_OP_FORWARD_BACKWARD, 1000, 64, 5000, LCE_BF16, LCE_RED_MEAN, LCE_BF16, 0);
  size_t b = lce_workspace_size(LCE_OP_FORWARD_BACKWARD, 4000, 64, 5000, LCE_BF16, LCE_RED_MEAN, LCE_BF16, 0);
  size_t c = lce_workspace_size(LCE_OP_FORWARD_BACKWARD, 4000, 64, 5000, LCE_BF16, LCE_RED_MEAN, LCE_BF16, 128);
  size_t f = lce_workspace_size(LCE_OP_FORWARD, 4000, 64, 5000, LCE_BF16, LCE_RED_MEAN, LCE_BF16, 0);
  size_t l = lce_workspace_size(LCE_OP_CE_FROM_LOGITS, 4000, 0, 5000, LCE_F32, LCE_RED_MEAN, LCE_F32, 0);
  CHECK(a > 0 && b > a && c > 0 && c < b && f > 0 && f < b && l > 0);
  CHECK(lce_workspace_size(LCE_OP_FORWARD, 10, 0, 10, LCE_F32, LCE_RED_MEAN, LCE_F32, 0) == 0); /* D < 1 */
  CHECK(lce_workspace_size(LCE_OP_FORWARD, 10, 8, 10, 7, LCE_RED_MEAN, LCE_F32, 0) == 0);       /* dtype */

  /* argument checks return before any launch (no GPU needed) */
  static int64_t target[4];
  static float loss[4];
  static unsigned char ws[1 << 12];
  void* fake = (void*)(uintptr_t)4096;
  CHECK(lce_forward(NULL, fake, NULL, target, 4, 8, 8, LCE_F32, LCE_F32, LCE_RED_MEAN, -100, loss, NULL, ws,
                    sizeof ws, NULL) == LCE_ERR_NULL);
  CHECK(lce_forward(fake, fake, NULL, target, 4, 8, 8, LCE_F32, LCE_BF16, LCE_RED_MEAN, -100, loss, NULL, ws,
                    sizeof ws, NULL) == LCE_ERR_DTYPE);
  CHECK(lce_forward(fake, fake, NULL, target, 4, 8, 8, LCE_F32, LCE_F32, 9, -100, loss, NULL, ws, sizeof ws,
                    NULL) == LCE_ERR_REDUCTION);
  CHECK(lce_forward_backward(fake, fake, NULL, target, 4, 8, 8, LCE_F32, LCE_F32, LCE_RED_NONE, -100, NULL, loss,
                             fake, fake, NULL, LCE_F32, ws, sizeof ws, NULL) == LCE_ERR_GRAD_OUT);
  CHECK(lce_forward(fake, fake, NULL, target, 4, 8, 8, LCE_F32, LCE_F32, LCE_RED_MEAN, -100, loss, NULL, NULL, 0,
                    NULL) == LCE_ERR_WORKSPACE);
  CHECK(lce_cross_entropy_from_logits(fake, target, 4, 0, LCE_F32, LCE_RED_MEAN, -100, NULL, loss, ws, sizeof ws,
                                      NULL) == LCE_ERR_SHAPE);
  CHECK(lce_cross_entropy_from_logits_noalloc(fake, target, (int64_t)LCE_NOALLOC_MAX_ROWS + 1, 8, LCE_F32,
                                              LCE_RED_MEAN, -100, NULL, loss, NULL, NULL) == LCE_ERR_SHAPE);
  CHECK(lce_test_gemm_bf16(NULL, fake, fake, 8, 8, 8, 0, 0, 0, NULL, NULL) == LCE_ERR_NULL);

  /* the bounded backward's plan: the default budget is 1 GiB of gradient
   * buffer; a larger budget stores more classes, a smaller one fewer */
  {
    const int64_t N = 8192, D = 4096, C = 128256;
    size_t def = lce_workspace_size(LCE_OP_FORWARD_BACKWARD, N, D, C, LCE_BF16, LCE_RED_MEAN, LCE_BF16, 0);
    size_t zero = lce_workspace_size_for_buffer(LCE_OP_FORWARD_BACKWARD, N, D, C, LCE_BF16, LCE_RED_MEAN, LCE_BF16, 0);
    size_t big = lce_workspace_size_for_buffer(LCE_OP_FORWARD_BACKWARD, N, D, C, LCE_BF16, LCE_RED_MEAN, LCE_BF16,
                                               (size_t)-1);
    size_t small = lce_workspace_size_for_buffer(LCE_OP_FORWARD_BACKWARD, N, D, C, LCE_BF16, LCE_RED_MEAN,
                                                 LCE_BF16, (size_t)256 << 20);
    CHECK(def == zero && big > def && small < def);
    CHECK(def < ((size_t)1 << 30) + ((size_t)256 << 20));
    int64_t plan[LCE_TEST_PLAN_FIELDS];
    CHECK(lce_test_plan(LCE_OP_FORWARD_BACKWARD, N, D, C, LCE_BF16, LCE_BF16, 1, 1, 0, def, plan,
                        LCE_TEST_PLAN_FIELDS) == LCE_TEST_PLAN_FIELDS);
    const int cb = LCE_TEST_PLAN_FIELDS - 3, cs = cb + 1, nvc = cb + 2; /* the last three fields */
    CHECK(plan[0] == N && plan[cb] == 65536 && plan[cs] == 65536 && plan[nvc] == 1); /* rows, Cb, Cs, chunks */
    size_t bw = lce_workspace_size(LCE_OP_BACKWARD, N, D, C, LCE_BF16, LCE_RED_NONE, LCE_BF16, 0);
    CHECK(lce_test_plan(LCE_OP_BACKWARD, N, D, C, LCE_BF16, LCE_BF16, 1, 1, 0, bw, plan,
                        LCE_TEST_PLAN_FIELDS) == LCE_TEST_PLAN_FIELDS);
    CHECK(plan[cs] == 0 && plan[nvc] == 2); /* lse given: nothing stored, two recomputed chunks */
  }

  /* gradients from a given lse, a given denominator, scaling: host checks */
  CHECK(lce_backward(fake, fake, NULL, target, NULL, 4, 8, 8, LCE_F32, LCE_F32, LCE_RED_MEAN, -100, NULL, fake,
                     fake, NULL, LCE_F32, ws, sizeof ws, NULL) == LCE_ERR_NULL); /* no lse */
  CHECK(lce_backward(fake, fake, NULL, target, (const float*)fake, 4, 8, 8, LCE_F32, LCE_F32, LCE_RED_NONE, -100,
                     NULL, fake, fake, NULL, LCE_F32, ws, sizeof ws, NULL) == LCE_ERR_GRAD_OUT);
  CHECK(lce_backward_ex(fake, fake, NULL, target, NULL, NULL, (const float*)fake, 4, 8, 8, LCE_F32, LCE_F32,
                        LCE_RED_MEAN, -100, NULL, fake, fake, NULL, 9, ws, sizeof ws, NULL) == LCE_ERR_DTYPE);
  CHECK(lce_forward_backward_ex(fake, fake, NULL, target, NULL, (const float*)fake, 4, 8, 8, LCE_F32, LCE_F32, 9,
                                -100, NULL, loss, fake, fake, NULL, LCE_F32, ws, sizeof ws, NULL) == LCE_ERR_REDUCTION);
  CHECK(lce_mean_denominator(target, NULL, 4, 8, -100, NULL, ws, sizeof ws, NULL) == LCE_ERR_NULL);
  CHECK(lce_mean_denominator(target, NULL, 4, 8, -100, loss, ws, 16, NULL) == LCE_ERR_WORKSPACE);
  CHECK(lce_scale_gradients(fake, 4, NULL, 0, NULL, 0, LCE_F32, NULL, NULL) == LCE_ERR_NULL);
  CHECK(lce_scale_gradients(fake, 4, NULL, 0, NULL, 0, 7, loss, NULL) == LCE_ERR_DTYPE);

  /* status strings and kernel accounting */
  for (int s = LCE_OK; s <= LCE_ERR_DEVICE; ++s) CHECK(lce_status_string(s) != NULL && strlen(lce_status_string(s)) > 0);
  CHECK(lce_num_kernel_ids() >= 10);
  CHECK(strcmp(lce_kernel_name(0), "prep") == 0);
  CHECK(lce_profile_reset() == LCE_OK);
  printf("C-ABI-OK\n");
  return 0;
}

/* Plain C client of the library: compiled and run by tests/test_c_abi.py (no GPU needed).
 * Exercises the host-only entry points and the argument checks through the C header. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "sa_api.h"

static int fails = 0;
#define CHECK(cond)                                          \
  do {                                                       \
    if (!(cond)) {                                           \
      fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
      ++fails;                                               \
    }                                                        \
  } while (0)

int main(void) {
  CHECK(sa_version() == 1);
  CHECK(strcmp(sa_status_string(SA_ERR_CAPACITY), "SA_ERR_CAPACITY") == 0);

  /* TOPK mask of the 8K workload: 2478 block pairs per sequence */
  sa_mask_params p;
  memset(&p, 0, sizeof(p));
  p.mode = SA_MASK_TOPK;
  p.block = 64;
  p.n_tokens = 8192;
  p.batch = 4;
  p.causal = 1;
  p.window_blocks = 4;
  p.global_blocks = 1;
  p.topk = 16;
  int64_t nnz = 0;
  CHECK(sa_mask_nnz_bound(&p, &nnz) == SA_OK);
  CHECK(nnz == 4 * 2478);
  p.components = SA_LITERAL_LOCAL; /* components belong to LITERAL_MEAN only */
  CHECK(sa_mask_nnz_bound(&p, &nnz) == SA_ERR_INVALID_ARG);

  /* Fibonacci offsets at alpha = 1, window 8, N = 1024: 13, 21, ..., 987 */
  int32_t offs[64];
  int32_t count = 0;
  CHECK(sa_fib_offsets(1, 1, 15, 8, 1024, offs, 64, &count) == SA_OK);
  CHECK(count == 10 && offs[0] == 13 && offs[9] == 987);
  CHECK(sa_fib_offsets(1, 1, 15, 8, 1024, offs, 2, &count) == SA_ERR_CAPACITY);

  /* coprime stagger: layer 1 of 16 takes ramp index 7, alpha = 1/2 + 7/15 = 29/30 */
  int32_t num = 0, den = 0;
  CHECK(sa_layer_alpha(1, 16, 1, 2, 3, 2, 7, &num, &den) == SA_OK);
  CHECK(num == 29 && den == 30);

  /* workspace size of the 8K backward */
  size_t ws = 0;
  CHECK(sa_attn_bwd_workspace_size(4, 8192, 12, 64, 4, 4 * 2478, &ws) == SA_OK);
  CHECK(ws >= (size_t)4 * 12 * 8192 * 4);

  /* per-block ratios of a constant byte run compress far below 1 */
  static uint8_t bytes[1024];
  memset(bytes, 'a', sizeof(bytes));
  float ratio[8];
  CHECK(sa_block_ratios(bytes, 1, 1024, 128, 6, ratio, 2) == SA_OK);
  for (int i = 0; i < 8; ++i) CHECK(ratio[i] > 0.f && ratio[i] < 0.25f);

  /* a compute call with a misaligned pointer is refused before any launch */
  const int64_t st[3] = {8192 * 12 * 64, 12 * 64, 64};
  CHECK(sa_attn_fwd((const void*)258, (const void*)256, (const void*)256, st, st, st, 1, 8192, 12, 12, 64, 64, 1,
                    (const int32_t*)256, (const int32_t*)256, 0, 0.125f, (void*)256, (float*)256, (void*)256, 4096,
                    NULL) == SA_ERR_UNSUPPORTED);
  /* the forward's workspace holds its work counter: at least 256 bytes */
  CHECK(sa_attn_fwd((const void*)256, (const void*)256, (const void*)256, st, st, st, 1, 8192, 12, 12, 64, 64, 1,
                    (const int32_t*)256, (const int32_t*)256, 0, 0.125f, (void*)256, (float*)256, (void*)256, 64,
                    NULL) == SA_ERR_CAPACITY);
  size_t fws = 0;
  CHECK(sa_attn_fwd_workspace_size(4, 8192, 12, 64, 64, 4, 1, &fws) == SA_OK && fws > 608 * 128 * 65 * 4);

  if (fails == 0) printf("c abi ok\n");
  return fails == 0 ? 0 : 1;
}

/* A C caller of libdllmcommit: the header compiles as C99 and the library
 * links and answers from C.  Only host-side entry points are called (no
 * device is needed); the test that builds and runs this program compares
 * what it prints with the oracle.
 *
 * Output, one item per line:
 *   version <string>
 *   status <code> <string>                      for every dllm_status
 *   ranges <P> <gen_len> <block_len> <align> <status> <n> <start end>...
 *   temperature <remaining> <num_steps> <bits of the fp32 result, hex>
 *   workspace <B> <L> <V> <dtype> <bytes>
 *   mask_bad_block_len <status>
 */
#include <inttypes.h>
#include <stdio.h>
#include <string.h>

#include "dllmcommit.h"

static void ranges(int64_t P, int64_t gen_len, int64_t block_len, int align) {
  int64_t r[2 * 64];
  int64_t n = -1;
  const dllm_status st = dllm_block_ranges(P, gen_len, block_len, align, r, 64, &n);
  printf("ranges %" PRId64 " %" PRId64 " %" PRId64 " %d %d %" PRId64, P, gen_len, block_len, align, (int)st, n);
  for (int64_t i = 0; st == DLLM_OK && i < n; ++i) printf(" %" PRId64 " %" PRId64, r[2 * i], r[2 * i + 1]);
  printf("\n");
}

static void temperature(int32_t remaining, int32_t num_steps) {
  float t = 0.0f;
  uint32_t bits = 0;
  const dllm_status st = dllm_linear_temperature(remaining, num_steps, 0.4f, 0.8f, &t);
  memcpy(&bits, &t, sizeof bits);
  printf("temperature %d %d %d %08x\n", (int)remaining, (int)num_steps, (int)st, (unsigned)bits);
}

int main(void) {
  printf("version %s\n", dllm_version());
  for (int s = DLLM_OK; s <= DLLM_ERR_DEVICE; ++s) {
    const char* msg = dllm_status_string((dllm_status)s);
    printf("status %d %s\n", s, msg ? msg : "(null)");
  }
  ranges(5, 70, 32, 0);
  ranges(5, 70, 32, 1);
  ranges(0, 64, 32, 1);
  ranges(7, 0, 32, 0);
  ranges(100, 1, 1, 0);
  temperature(0, 48);
  temperature(17, 48);
  temperature(48, 48);
  printf("workspace 1 32 126464 %d %zu\n", (int)DLLM_BF16, dllm_token_stats_workspace_size(1, 32, 126464, DLLM_BF16));
  printf("mask_bad_block_len %d\n",
         (int)dllm_block_causal_mask(4, 4, 0, 0, 0, DLLM_MASK_F32, NULL, 4, (dllm_stream_t)0));
  return 0;
}

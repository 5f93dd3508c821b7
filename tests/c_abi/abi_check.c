/* A plain C11 consumer of include/pa.h and libpa.so. It makes only the calls that
 * need no GPU (version, status strings, argument validation, the launch plan) and
 * prints one line per check for tests/test_c_abi.py to read. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "pa.h"

static pa_decode_args base_args(void) {
  pa_decode_args a;
  memset(&a, 0, sizeof a);
  a.q = (const void*)16;
  a.k_cache = (const void*)32;
  a.v_cache = (const void*)48;
  a.block_tables = (const int32_t*)64;
  a.seq_lens = (const int32_t*)80;
  a.out = (void*)96;
  a.B = 1;
  a.Hq = 24;
  a.Hkv = 4;
  a.D = 256;
  a.block_size = 784;
  a.num_blocks = 64;
  a.max_blocks_per_seq = 42;
  a.max_seq_len = 32768;
  a.scale = 0.0625f;
  a.dtype = PA_BF16;
  return a;
}

int main(void) {
  printf("version %s\n", pa_version());
  printf("status %d %s\n", (int)PA_ERR_WORKSPACE, pa_status_string(PA_ERR_WORKSPACE));

  pa_decode_args a = base_args();
  int splits = 0, tokens = 0;
  pa_status st = pa_decode_plan(&a, 152, &splits, &tokens);
  printf("plan %d %d %d\n", (int)st, splits, tokens);

  a.Hq = 25; /* not a multiple of Hkv */
  printf("invalid %d\n", (int)pa_decode_ex(&a, (void*)256, 1u << 20, NULL));

  a = base_args();
  a.flags = PA_FLAG_DETERMINISTIC;
  printf("deterministic_plan %d\n", (int)pa_decode_plan(&a, 152, &splits, &tokens));

  printf("header_bytes %u\n", (unsigned)PA_WORKSPACE_HEADER_BYTES);
  return 0;
}

/* A plain C11 program that runs one paged decode through include/pa.h on the GPU:
 * B = 2 sequences (1000 and 37 tokens), 8 query / 2 KV heads, head_dim 128,
 * block 16, bf16 values from a 64-bit linear congruential generator, blocks taken
 * in a shuffled order from a 160-block pool. It writes q, each sequence's K and V
 * in token order (as generated, before paging), the lengths and the output to one
 * binary file for tests/test_c_abi.py, which checks the output against the float64
 * oracle. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "pa.h"

enum { B = 2, HQ = 8, HKV = 2, D = 128, BS = 16, NB = 160, MAXB = 63 };
static const int LENS[B] = {1000, 37};

static uint64_t rng = 0x9E3779B97F4A7C15ull;
static uint32_t next_u32(void) {
  rng = rng * 6364136223846793005ull + 1442695040888963407ull;
  return (uint32_t)(rng >> 32);
}
/* bf16 bits of a value in [-2, 2): the top half of an fp32 */
static uint16_t next_bf16(void) {
  const float x = ((float)(next_u32() >> 8) / 16777216.0f) * 4.0f - 2.0f;
  uint32_t u;
  memcpy(&u, &x, 4);
  return (uint16_t)(u >> 16);
}

#define CHECK(x)                                                         \
  do {                                                                   \
    if ((x) != cudaSuccess) {                                            \
      fprintf(stderr, "CUDA error at %s:%d\n", __FILE__, __LINE__);      \
      return 2;                                                          \
    }                                                                    \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 2) return 1;
  const size_t nq = (size_t)B * HQ * D, nkv = (size_t)NB * BS * HKV * D;
  uint16_t* q = malloc(nq * 2);
  uint16_t* k = calloc(nkv, 2);
  uint16_t* v = calloc(nkv, 2);
  uint16_t* out = malloc(nq * 2);
  uint16_t* kc = malloc((size_t)(LENS[0] + LENS[1]) * HKV * D * 2);  /* token order */
  uint16_t* vc = malloc((size_t)(LENS[0] + LENS[1]) * HKV * D * 2);
  int32_t bt[B * MAXB], sl[B], perm[NB];
  for (size_t i = 0; i < nq; ++i) q[i] = next_bf16();
  for (int i = 0; i < NB; ++i) perm[i] = i;
  for (int i = NB - 1; i > 0; --i) {  /* Fisher-Yates */
    const int j = (int)(next_u32() % (uint32_t)(i + 1)), t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
  int used = 0;
  size_t tc = 0;  /* tokens written in token order so far */
  for (int b = 0; b < B; ++b) {
    sl[b] = LENS[b];
    for (int j = 0; j < MAXB; ++j) bt[b * MAXB + j] = -1;
    for (int j = 0; j < (LENS[b] + BS - 1) / BS; ++j) bt[b * MAXB + j] = perm[used++];
    for (int t = 0; t < LENS[b]; ++t, ++tc) {
      const size_t row = ((size_t)bt[b * MAXB + t / BS] * BS + t % BS) * HKV;
      for (size_t e = 0; e < (size_t)HKV * D; ++e) {
        kc[tc * HKV * D + e] = next_bf16();
        vc[tc * HKV * D + e] = next_bf16();
        k[row * D + e] = kc[tc * HKV * D + e];
        v[row * D + e] = vc[tc * HKV * D + e];
      }
    }
  }
  void *dq, *dk, *dv, *dbt, *dsl, *dout, *ws;
  const size_t wsb = pa_decode_workspace_bytes(B, HQ, HKV, D, 1000);
  if (wsb == 0) return 3;
  CHECK(cudaMalloc(&dq, nq * 2));
  CHECK(cudaMalloc(&dk, nkv * 2));
  CHECK(cudaMalloc(&dv, nkv * 2));
  CHECK(cudaMalloc(&dbt, sizeof bt));
  CHECK(cudaMalloc(&dsl, sizeof sl));
  CHECK(cudaMalloc(&dout, nq * 2));
  CHECK(cudaMalloc(&ws, wsb));
  CHECK(cudaMemcpy(dq, q, nq * 2, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dk, k, nkv * 2, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dv, v, nkv * 2, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dbt, bt, sizeof bt, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dsl, sl, sizeof sl, cudaMemcpyHostToDevice));
  if (pa_workspace_init(ws, wsb, NULL) != PA_OK) return 4;
  const pa_status st = pa_decode(dq, dk, dv, (const int32_t*)dbt, (const int32_t*)dsl, dout, B,
                                 HQ, HKV, D, BS, NB, MAXB, 1000, 0.08838834764831845f, PA_BF16,
                                 ws, wsb, NULL);
  if (st != PA_OK) {
    fprintf(stderr, "pa_decode: %s\n", pa_status_string(st));
    return 5;
  }
  uint32_t flags = 1;
  if (pa_read_device_errors(ws, NULL, &flags) != PA_OK || flags != 0) return 6;
  CHECK(cudaMemcpy(out, dout, nq * 2, cudaMemcpyDeviceToHost));
  FILE* f = fopen(argv[1], "wb");
  if (!f) return 7;
  fwrite(q, 2, nq, f);
  fwrite(kc, 2, tc * HKV * D, f);
  fwrite(vc, 2, tc * HKV * D, f);
  fwrite(sl, 4, B, f);
  fwrite(out, 2, nq, f);
  fclose(f);
  printf("ok\n");
  return 0;
}

// Launch parameters shared by the host launcher and the decode kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "pa.h"

namespace pa {

// Split counts are bounded, so that the partials stay a small fraction of the KV
// bytes at any context length.
constexpr int kMaxSplits = 1024;
constexpr int kPartitionMin = 64;   // tokens: below this a split's fixed cost dominates
// Tokens per warp tile (a multiple of the score MMA's 16 rows); split partitions
// and static shares are whole tiles.
#ifndef PA_TILE_TOKENS_D128
#define PA_TILE_TOKENS_D128 32
#endif
#ifndef PA_TILE_TOKENS_D256
#define PA_TILE_TOKENS_D256 16
#endif
#ifndef PA_TILE_TOKENS_F8_D128
#define PA_TILE_TOKENS_F8_D128 32
#endif
#ifndef PA_TILE_TOKENS_F8_D256
#define PA_TILE_TOKENS_F8_D256 32
#endif
// Per head_dim and cache type: a 256-wide 16-bit row pair is already 1 KB a token;
// fp8 rows carry half the bytes of a 16-bit row for the same arithmetic.
constexpr int tile_tokens(int D, bool fp8) {
  return fp8 ? (D == 128 ? PA_TILE_TOKENS_F8_D128 : PA_TILE_TOKENS_F8_D256)
             : (D == 128 ? PA_TILE_TOKENS_D128 : PA_TILE_TOKENS_D256);
}
// Warps per decode CTA, per head_dim and cache type: fp8 tiles cost more math per
// byte, so the fp8 kernel at head_dim 128 runs more warps.
#ifndef PA_WARPS_D128
#define PA_WARPS_D128 4
#endif
#ifndef PA_WARPS_D256
#define PA_WARPS_D256 4
#endif
#ifndef PA_WARPS_F8_D128
#define PA_WARPS_F8_D128 8
#endif
#ifndef PA_WARPS_F8_D256
#define PA_WARPS_F8_D256 4
#endif
constexpr int warps_per_cta(int D, bool fp8) {
  return D == 128 ? (fp8 ? PA_WARPS_F8_D128 : PA_WARPS_D128) : (fp8 ? PA_WARPS_F8_D256 : PA_WARPS_D256);
}
// Work sharing among the splits of a sequence: each split keeps about
// (1 - 1/kStealDiv) of its P tokens as a static share, and the rest of the context
// is claimed tile by tile through one counter per (sequence, KV head) held in the
// workspace header, for up to kStealUnits such pairs (beyond that, static splits)
// and for splits that stream at least kStealMinBytes.
#ifndef PA_STEAL_DIV
#define PA_STEAL_DIV 8
#endif
constexpr int kStealDiv = PA_STEAL_DIV;
// Shorter splits stay static: their imbalance costs less than a claim's round trip.
#ifndef PA_STEAL_MIN_KIB
#define PA_STEAL_MIN_KIB 512
#endif
constexpr long long kStealMinBytes = (long long)PA_STEAL_MIN_KIB * 1024;  // K + V bytes per split
constexpr int kStealUnits = 2048;
// Largest split count whose splits merge inside their thread-block cluster (the
// portable cluster size).
constexpr int kMaxClusterMerge = 8;
constexpr int kHeaderBytes = 256 + kStealUnits * 4;  // error word, then the counters
static_assert(kHeaderBytes % 256 == 0, "header keeps 256-byte alignment");
static_assert(kHeaderBytes == PA_WORKSPACE_HEADER_BYTES, "header size is part of the ABI");

struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  void* out;
  float* ws_m;        // [B*Hkv*S][G]   running max of each split (log2 domain)
  float* ws_l;        // [B*Hkv*S][G]   softmax denominator of each split
  float* ws_acc;      // [B*Hkv*S][G][D] unnormalised output of each split
  uint32_t* err;      // device error word
  int* steal;         // [B*Hkv] claimed shared tiles per (sequence, KV head); zero between calls
  int B, Hq, Hkv, G;
  int block_size, num_blocks, max_blocks, max_seq_len;
  // t / block_size for 0 <= t < 2^31 without a division: (t >> bs_shift) for a
  // power of two (bs_magic == 0), else umulhi(t, bs_magic) >> bs_shift
  uint32_t bs_magic;
  int bs_shift;
  int S, P;           // splits and tokens per split
  int Ps;             // static tokens per split (== P: no shared tiles)
  int window;         // > 0: attend to the last `window` tokens only
  int q_len;          // query rows per sequence (causal among themselves)
  int kv_fp8;         // caches hold FP8 E4M3 (k_scale is folded into scale_log2)
  int cmerge;         // 0, or C = S: the S splits of each (sequence, KV head) run as one
                      // thread-block cluster and merge in distributed shared memory (set
                      // by the launcher; no merge grid)
  float v_scale;      // cache V value = stored value * v_scale
  float scale_log2;   // scale * log2(e): scores live in the exp2 domain
};

// One launcher per (dtype, head_dim); each dispatches on the GQA group size. With
// kernels != nullptr nothing is launched: *kernels is set to the number of kernels
// the launch would make (1, or 2 with a merge grid).
cudaError_t launch_decode_bf16_d128(const DecodeParams& p, cudaStream_t st, int* kernels = nullptr);
cudaError_t launch_decode_bf16_d256(const DecodeParams& p, cudaStream_t st, int* kernels = nullptr);
cudaError_t launch_decode_f16_d128(const DecodeParams& p, cudaStream_t st, int* kernels = nullptr);
cudaError_t launch_decode_f16_d256(const DecodeParams& p, cudaStream_t st, int* kernels = nullptr);
// FP8 E4M3 caches with bf16 / fp16 queries and outputs.
cudaError_t launch_decode_fp8_bf16_d128(const DecodeParams& p, cudaStream_t st, int* kernels = nullptr);
cudaError_t launch_decode_fp8_bf16_d256(const DecodeParams& p, cudaStream_t st, int* kernels = nullptr);
cudaError_t launch_decode_fp8_f16_d128(const DecodeParams& p, cudaStream_t st, int* kernels = nullptr);
cudaError_t launch_decode_fp8_f16_d256(const DecodeParams& p, cudaStream_t st, int* kernels = nullptr);

}  // namespace pa

// Decode kernels for FP8 E4M3 caches with f16 queries, head_dim 128.
#include "pa_decode_kernel.cuh"

namespace pa {
cudaError_t launch_decode_fp8_f16_d128(const DecodeParams& p, cudaStream_t st, int* kernels) {
  return launch_decode_dispatch<__half, fp8e4m3, 128>(p, st, kernels);
}
}  // namespace pa

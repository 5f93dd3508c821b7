// Decode kernels for f16 caches with head_dim 128.
#include "pa_decode_kernel.cuh"

namespace pa {
cudaError_t launch_decode_f16_d128(const DecodeParams& p, cudaStream_t st, int* kernels) {
  return launch_decode_dispatch<__half, __half, 128>(p, st, kernels);
}
}  // namespace pa

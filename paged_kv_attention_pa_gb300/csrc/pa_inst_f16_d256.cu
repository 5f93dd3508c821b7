// Decode kernels for f16 caches with head_dim 256.
#include "pa_decode_kernel.cuh"

namespace pa {
cudaError_t launch_decode_f16_d256(const DecodeParams& p, cudaStream_t st, int* kernels) {
  return launch_decode_dispatch<__half, __half, 256>(p, st, kernels);
}
}  // namespace pa

// Decode kernels for bf16 caches with head_dim 128.
#include "pa_decode_kernel.cuh"

namespace pa {
cudaError_t launch_decode_bf16_d128(const DecodeParams& p, cudaStream_t st, int* kernels) {
  return launch_decode_dispatch<__nv_bfloat16, __nv_bfloat16, 128>(p, st, kernels);
}
}  // namespace pa

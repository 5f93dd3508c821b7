// pa_decode_noalloc: the decode call for callers that cannot provide a workspace.
//
// Some callers have no way to hand this library device scratch memory: a plugin
// living inside another runtime that owns every device allocation, code that
// must never call cudaMalloc (it can synchronise the whole device), or a thin
// binding with no device allocator of its own. For them this file keeps the
// split partials in one fixed array that is part of the library's device image,
// so the call itself allocates nothing. The array costs every GPU that loads this
// module PA_NOALLOC_SCRATCH_BYTES of memory until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "pa.h"

// Device scratch shared by every pa_decode_noalloc call on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};  // device address of the array, per device

// Once per device, with that device current: look up the array's device address
// (the host-side name is only a stand-in, never a device pointer). The array is
// zero when the module loads; its header (the device error word and the tile
// counters) is cleared once more on the caller's stream before the first launch,
// so that the clearing is ordered before that launch whatever the stream.
pa_status scratch_for_current_device(cudaStream_t stream, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    if (cudaMemsetAsync(addr, 0, PA_WORKSPACE_HEADER_BYTES, stream) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* seq_lens,
                                       void* out, int B, int Hq, int Hkv, int D, int block_size,
                                       int num_blocks, int max_blocks_per_seq, int max_seq_len,
                                       float scale, pa_dtype dtype, pa_stream_t stream) {
  pa_decode_args a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.out = out;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_seq_len = max_seq_len;
  a.scale = scale;
  a.dtype = dtype;
  a.splits = 0;
  if (B == 0) return pa_decode_ex(&a, nullptr, 0, stream);  // validation only, no launch
  const size_t need = pa_decode_ex_workspace_bytes(&a);
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;  // too big for the array
  if (need == 0) {
    // invalid sizes (reported by pa_decode_ex, which launches nothing without a
    // workspace), or no usable device
    const pa_status st = pa_decode_ex(&a, nullptr, 0, stream);
    return st == PA_ERR_WORKSPACE ? PA_ERR_CUDA : st;
  }
  void* scratch = nullptr;
  const pa_status st = scratch_for_current_device((cudaStream_t)stream, &scratch);
  if (st != PA_OK) return st;
  return pa_decode_ex(&a, scratch, PA_NOALLOC_SCRATCH_BYTES, stream);
}

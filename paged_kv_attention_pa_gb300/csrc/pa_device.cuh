// Device-side helpers for sm_103a: L2 cache policy, fp8 widening, dependent-launch
// and cluster primitives, 16-bit float packing, and the warp-level MMA / ldmatrix /
// movmatrix wrappers. Inline PTX only; no library code.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace pa {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// L2 policy for data read exactly once (the KV stream): evict first, so that the
// small split partials stay resident.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// ---------------------------------------------------------------- fp8 caches
// Tag type of an FP8 E4M3 cache element (one byte: sign, 4-bit exponent with bias
// 7, 3-bit mantissa; no infinities).
struct fp8e4m3 {
  uint8_t bits;
};

// Two E4M3 values (low byte = element 0) to a packed pair of fp16, exactly: every
// E4M3 value is representable in fp16.
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint16_t x) {
  uint32_t y;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(y) : "h"(x));
  return y;
}

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32, relative error about
// 2^-22). Every use here has x <= 0 (softmax weights, rescale factors): results lie
// in [0, 1], subnormal ones flush to zero, and 2^-inf = +0.
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Ask for the L2 line holding p (no data returned; a hint the memory system may drop).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// 16-byte shared-memory load from a shared-window address.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
// Word i (0..3) of a 16-byte vector; i is a constant after unrolling.
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// ---------------------------------------------------------------- dependent launch
// Wait until the grids this one depends on (programmatic launch) have completed
// and their writes are visible; returns at once for an ordinary launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Thread-block cluster barrier (all threads of every CTA of the cluster): a hardware
// barrier; release / acquire order the shared-memory writes before it (to this CTA's
// memory or another's of the cluster) before every access after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// Cluster barrier that orders execution only (relaxed arrive): for handing over
// memory that no thread of the cluster has accesses pending on.
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" :::
                   "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Generic address of the same shared-memory object in CTA `rank` of this cluster:
// plain loads and stores through it reach that CTA's shared memory (distributed
// shared memory) and are scheduled like any other memory access.
__device__ __forceinline__ const float* map_cluster_rank(const float* p, uint32_t rank) {
  uint64_t r;
  asm volatile("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(p), "r"(rank));
  return reinterpret_cast<const float*>(r);
}
// Allow the next grid in the stream to be scheduled (it still waits in pdl_wait).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- 16-bit unpack
// Two packed 16-bit floats (low half = element 0) to two fp32 values, exactly.
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);

template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
  // bf16 is the top half of an fp32: shift / mask, no rounding involved.
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) {
  return __float2half_rn(x);
}

// ---------------------------------------------------------------- warp MMA
// m16n8k16 fragments (PTX ISA, warp-level matrix fragments): with gid = lane / 4
// and tig = lane % 4, A holds rows {gid, gid+8} x cols {2tig, 2tig+1, 2tig+8,
// 2tig+9}, B holds rows {2tig, 2tig+1, 2tig+8, 2tig+9} x col gid, C holds rows
// {gid, gid+8} x cols {2tig, 2tig+1}.
template <typename T>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);

template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&c)[4], const uint32_t (&a)[4],
                                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <>
__device__ __forceinline__ void mma16816<__half>(float (&c)[4], const uint32_t (&a)[4],
                                                 uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 16-bit matrices from shared memory; lane i gives the row address of
// row i % 8 of matrix i / 8. TRANS loads each matrix transposed.
template <bool TRANS>
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  if constexpr (TRANS)
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
  else
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// Transpose an 8x8 16-bit matrix held in fragment layout across the warp.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Two fp32 values to one packed pair (lo in the low half), round to nearest even.
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace pa

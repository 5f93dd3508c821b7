// Split-KV single-query paged-attention decode for sm_103a.
//
// One CTA serves one (split, KV head, sequence): all G query heads of that KV
// head share every K/V tile it stages ("one workgroup per (sequence, KV head)"
// in "Hybrid-SSM decode rate on dual Radeon cards under vLLM", widened by the
// split-KV fix of the same page so that B * Hkv * splits fills every SM even at
// batch 1 with 4 KV heads).
//
// Warp roles inside a CTA:
//   warp NW (producer)  stages the CTA's block-table slice, then streams K/V
//                       rows into a ring of shared-memory stages with 1-D bulk
//                       copies (TMA engine, one row of D elements each), each
//                       stage completing on an mbarrier as transaction bytes.
//                       Only rows of live tokens (t < seq_len) are copied: the
//                       unwritten tail of the last block is never read
//                       ("vLLM's custom ROCm paged-attention kernel wins all
//                       sixty cells", §5, the V-load fault).
//   warps 0..NW-1       consume warp tiles round-robin. Scores: lane-per-token,
//   (consumers)         q broadcast from shared memory, packed fp32x2 FMAs,
//                       tokens past seq_len set to -inf by select. Online
//                       softmax in the exp2 domain with warp-shuffle maxima.
//                       PV: lane-per-output-element, p broadcast from shared
//                       memory; the loop stops at the last live token, so V rows
//                       past seq_len never reach the accumulator.
// Epilogue: the consumer warps merge their (m, l, acc) in shared memory. A single
// split writes the output; otherwise the split's partial goes to the workspace
// and the last CTA of the (sequence, KV head) to finish (atomic counter, no
// waiting) merges all partials and writes the output.
#pragma once

#include <cstdint>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_params.h"

namespace pa {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kSmemBudget = 220 * 1024;
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s: only a logic error gets here
constexpr int kMergeBar = 1;                           // named barrier id for consumers

template <int D, int GT>
struct Cfg {
  static constexpr int LPT = D / 128;           // lanes per token in the score phase
  static constexpr int TW = 32 / LPT;           // tokens per warp tile
  static constexpr int ROWB = D * 2 + 16;       // smem row pitch, padded against bank conflicts
  static constexpr int TILE_BYTES = TW * ROWB;  // K (or V) half of a stage
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int DPL = D / 32;            // output elements per lane in the PV phase
  static constexpr int GP = (GT + 3) / 4 * 4;   // pitch of a token's p row (floats)
  static constexpr int QH = D / LPT;            // q elements a lane's score covers
  static constexpr int QROW = QH + 4;           // padded q half-row (floats)
  static constexpr int CHAINS = GT <= 4 ? 2 : 1;  // independent FMA chains per head
  static constexpr int Q_BYTES = GT * LPT * QROW * 4;
  static constexpr int P_BYTES = kConsumerWarps * TW * GP * 4;
  static constexpr int BT_BYTES = kBtMax * 4;
  static constexpr int FIXED = Q_BYTES + P_BYTES + BT_BYTES + 512;
  static constexpr int NS_FIT = (kSmemBudget - FIXED) / STAGE_BYTES;
  static constexpr int NS = NS_FIT > 12 ? 12 : NS_FIT;
  static constexpr int SMEM = NS * STAGE_BYTES + FIXED;
  static constexpr int RING = NS * STAGE_BYTES;
  static_assert(NS >= 2 * kConsumerWarps, "need at least two stages per consumer warp");
  static_assert(kConsumerWarps * GT * (D + 2) * 4 <= RING, "CTA merge must fit in the ring");
  static_assert((kMaxSplits + 2) * GT * 4 <= RING, "split merge must fit in the ring");
};

template <typename T, int D, int GT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
  using C = Cfg<D, GT>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* q_s = reinterpret_cast<float*>(smem + C::RING);
  float* p_s = reinterpret_cast<float*>(smem + C::RING + C::Q_BYTES);
  int* bt_s = reinterpret_cast<int*>(smem + C::RING + C::Q_BYTES + C::P_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::RING + C::Q_BYTES + C::P_BYTES +
                                               C::BT_BYTES);
  uint64_t* empty = full + C::NS;
  int* flag_s = reinterpret_cast<int*>(empty + C::NS);

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  T* out = reinterpret_cast<T*>(p.out);
  const size_t head0 = (size_t)b * p.Hq + (size_t)kvh * G;

  // ---- context length, validated against the bounds the launch was planned for
  int L = __ldg(p.seq_lens + b);
  {
    const long long cap_ll = (long long)p.max_blocks * p.block_size;
    const int cap = (int)min((long long)p.max_seq_len, cap_ll);
    if (L < 0 || L > cap) {
      if (split == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_SEQ_LEN);
      L = L < 0 ? 0 : cap;
    }
  }
  if (L == 0) {  // empty context: a zero row, written once
    if (split == 0)
      for (int i = threadIdx.x; i < G * D; i += kThreads) out[head0 * D + i] = from_f32<T>(0.f);
    return;
  }
  const int t_begin = split * p.P;
  if (t_begin >= L) return;  // this split lies past the sequence: nothing to do
  const int t_end = min(L, t_begin + p.P);
  const int n_tiles = (t_end - t_begin + C::TW - 1) / C::TW;
  const int n_splits = (L + p.P - 1) / p.P;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ================================================================ producer
    const int blk0 = t_begin / p.block_size;
    int nb = (t_end - 1) / p.block_size - blk0 + 1;
    if (nb > kBtMax) {  // the planner never allows this; stay in bounds regardless
      if (lane == 0) atomicOr(p.err, PA_DEVERR_SEQ_LEN);
      nb = kBtMax;
    }
    const int32_t* bt_row = p.block_tables + (size_t)b * p.max_blocks;
    for (int i = lane; i < nb; i += 32) {
      int phys = __ldg(bt_row + blk0 + i);
      if (phys < 0 || phys >= p.num_blocks) {
        atomicOr(p.err, PA_DEVERR_BLOCK_INDEX);
        phys = 0;
      }
      bt_s[i] = phys;
    }
    __syncwarp();
    const uint64_t pol = l2_evict_first_policy();
    const T* kbase = reinterpret_cast<const T*>(p.k_cache);
    const T* vbase = reinterpret_cast<const T*>(p.v_cache);
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % C::NS;
      const uint32_t par = ((j / C::NS) & 1) ^ 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&empty[s], par, kWaitLimitCycles);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) atomicOr(p.err, PA_DEVERR_TIMEOUT);
        break;
      }
      const int t0 = t_begin + j * C::TW;
      const int nv = min(C::TW, t_end - t0);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(nv * 2 * D * sizeof(T)));
      __syncwarp();
      if (lane < nv) {
        const int t = t0 + lane;
        const int lb = t / p.block_size;
        const int off = t - lb * p.block_size;
        const int idx = min(lb - blk0, nb - 1);
        const size_t row = ((size_t)bt_s[idx] * p.block_size + off) * p.Hkv + kvh;
        uint8_t* dk = ring + s * C::STAGE_BYTES + lane * C::ROWB;
        bulk_g2s(dk, kbase + row * D, D * sizeof(T), &full[s], pol);
        bulk_g2s(dk + C::TILE_BYTES, vbase + row * D, D * sizeof(T), &full[s], pol);
      }
      issued = j + 1;
    }
    // Do not leave while copies into this CTA's shared memory may be in flight.
    if (lane == 0) {
      const int first = issued > C::NS ? issued - C::NS : 0;
      for (int j = first; j < issued; ++j)
        if (!mbar_wait_bounded(&full[j % C::NS], (j / C::NS) & 1, kWaitLimitCycles)) {
          atomicOr(p.err, PA_DEVERR_TIMEOUT);
          break;
        }
    }
    return;
  }

  // ================================================================== consumers
  const int ctid = threadIdx.x;  // 0 .. kConsumerThreads-1
  {
    const T* qg = reinterpret_cast<const T*>(p.q) + head0 * D;
    for (int i = ctid; i < GT * D; i += kConsumerThreads) {
      const int g = i / D, d = i - (i / D) * D;
      const float v = g < G ? to_f32<T>(qg[(size_t)g * D + d]) * p.scale_log2 : 0.f;
      const int hf = d / C::QH, dd = d - hf * C::QH;
      q_s[(g * C::LPT + hf) * C::QROW + dd] = v;
    }
  }
  named_bar_sync(kMergeBar, kConsumerThreads);

  const int r = lane % C::TW;   // token of the warp tile this lane scores
  const int hf = lane / C::TW;  // which half of D (head_dim 256 only)
  float m[GT], l[GT];
  float2 acc[GT][C::DPL / 2];
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < C::DPL / 2; ++i) acc[g][i] = make_float2(0.f, 0.f);
  }
  float* pw = p_s + warp * C::TW * C::GP;

  for (int j = warp; j < n_tiles; j += kConsumerWarps) {
    const int s = j % C::NS;
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(&full[s], (j / C::NS) & 1, kWaitLimitCycles);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) atomicOr(p.err, PA_DEVERR_TIMEOUT);
      break;
    }
    const int nv = min(C::TW, t_end - (t_begin + j * C::TW));
    const uint8_t* kt = ring + s * C::STAGE_BYTES;
    const uint8_t* vt = kt + C::TILE_BYTES;

    // ---- scores s[g] = (scale*log2e*q_g) . k_r over this lane's part of D
    float sc[GT];
    {
      float2 a[C::CHAINS][GT];
#pragma unroll
      for (int c = 0; c < C::CHAINS; ++c)
#pragma unroll
        for (int g = 0; g < GT; ++g) a[c][g] = make_float2(0.f, 0.f);
      const uint8_t* krow = kt + r * C::ROWB + hf * (C::QH * 2);
#pragma unroll
      for (int c = 0; c < C::QH / 8; ++c) {
        const uint4 kw = *reinterpret_cast<const uint4*>(krow + c * 16);
        const float2 k0 = unpack2<T>(kw.x), k1 = unpack2<T>(kw.y);
        const float2 k2 = unpack2<T>(kw.z), k3 = unpack2<T>(kw.w);
#pragma unroll
        for (int g = 0; g < GT; ++g) {
          const float* qr = q_s + (g * C::LPT + hf) * C::QROW + c * 8;
          const float4 qa = *reinterpret_cast<const float4*>(qr);
          const float4 qb = *reinterpret_cast<const float4*>(qr + 4);
          a[0][g] = ffma2(make_float2(qa.x, qa.y), k0, a[0][g]);
          a[C::CHAINS - 1][g] = ffma2(make_float2(qa.z, qa.w), k1, a[C::CHAINS - 1][g]);
          a[0][g] = ffma2(make_float2(qb.x, qb.y), k2, a[0][g]);
          a[C::CHAINS - 1][g] = ffma2(make_float2(qb.z, qb.w), k3, a[C::CHAINS - 1][g]);
        }
      }
      const bool live = r < nv;
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        float v = a[0][g].x + a[0][g].y;
        if (C::CHAINS == 2) v += a[C::CHAINS - 1][g].x + a[C::CHAINS - 1][g].y;
        if (C::LPT == 2) v += __shfl_xor_sync(0xffffffffu, v, 16);
        sc[g] = live ? v : -INFINITY;  // select, so garbage or NaN in a dead row is dropped
      }
    }

    // ---- online softmax (exp2 domain); p goes to shared memory for the PV phase
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      float mt = sc[g];
#pragma unroll
      for (int o = C::TW / 2; o >= 1; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float mn = fmaxf(m[g], mt);
      const float mref = mn == -INFINITY ? 0.f : mn;
      const float alpha = exp2f(m[g] - mref);
      const float pv = exp2f(sc[g] - mref);
      l[g] = l[g] * alpha + (hf == 0 ? pv : 0.f);
      m[g] = mn;
      const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
      for (int i = 0; i < C::DPL / 2; ++i) acc[g][i] = fmul2(acc[g][i], a2);
      if (hf == 0) pw[r * C::GP + g] = pv;
    }
    __syncwarp();

    // ---- acc[g][:] += p[g][t] * v_t over live tokens only
    const uint8_t* vcol = vt + lane * (C::DPL * 2);
#pragma unroll 2
    for (int t = 0; t < nv; ++t) {
      float2 vv[C::DPL / 2];
      if constexpr (C::DPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(vcol + t * C::ROWB);
        vv[0] = unpack2<T>(w.x);
        vv[1] = unpack2<T>(w.y);
      } else {
        const uint4 w = *reinterpret_cast<const uint4*>(vcol + t * C::ROWB);
        vv[0] = unpack2<T>(w.x);
        vv[1] = unpack2<T>(w.y);
        vv[2] = unpack2<T>(w.z);
        vv[3] = unpack2<T>(w.w);
      }
      const float* pr = pw + t * C::GP;
#pragma unroll
      for (int g4 = 0; g4 < C::GP / 4; ++g4) {
        const float4 p4 = *reinterpret_cast<const float4*>(pr + g4 * 4);
        const float pg[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int g = g4 * 4 + k;
          if (g < GT) {
            const float2 pp = make_float2(pg[k], pg[k]);
#pragma unroll
            for (int i = 0; i < C::DPL / 2; ++i) acc[g][i] = ffma2(pp, vv[i], acc[g][i]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- denominators: sum the per-lane partial sums
#pragma unroll
  for (int g = 0; g < GT; ++g)
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) l[g] += __shfl_xor_sync(0xffffffffu, l[g], o);

  // ---- merge the consumer warps (the ring is free: every tile was consumed)
  named_bar_sync(kMergeBar, kConsumerThreads);
  float* mw = reinterpret_cast<float*>(ring);  // [NW][GT]
  float* lw = mw + kConsumerWarps * GT;        // [NW][GT]
  float* aw = lw + kConsumerWarps * GT;        // [NW][GT][D]
  if (lane == 0)
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      mw[warp * GT + g] = m[g];
      lw[warp * GT + g] = l[g];
    }
#pragma unroll
  for (int g = 0; g < GT; ++g)
#pragma unroll
    for (int i = 0; i < C::DPL / 2; ++i)
      *reinterpret_cast<float2*>(aw + (warp * GT + g) * D + lane * C::DPL + 2 * i) = acc[g][i];
  named_bar_sync(kMergeBar, kConsumerThreads);

  const bool single = n_splits == 1;
  const size_t pidx = ((size_t)b * p.Hkv + kvh) * p.S + split;
  for (int i = ctid; i < G * D; i += kConsumerThreads) {
    const int g = i / D, d = i - (i / D) * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mw[w * GT + g]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float e = exp2f(mw[w * GT + g] - M);  // idle warps: m = -inf, weight 0
      num += e * aw[(w * GT + g) * D + d];
      den += e * lw[w * GT + g];
    }
    if (single) {
      out[(head0 + g) * D + d] = from_f32<T>(num / den);
    } else {
      p.ws_acc[(pidx * G + g) * D + d] = num;
      if (d == 0) {
        p.ws_m[pidx * G + g] = M;
        p.ws_l[pidx * G + g] = den;
      }
    }
  }
  if (single) return;

  // ---- split merge by whichever CTA of this (sequence, KV head) finishes last
  __threadfence();
  named_bar_sync(kMergeBar, kConsumerThreads);
  if (ctid == 0) {
    const uint32_t done = atomicAdd(p.counters + (size_t)b * p.Hkv + kvh, 1u);
    flag_s[0] = done == (uint32_t)(n_splits - 1);
  }
  named_bar_sync(kMergeBar, kConsumerThreads);
  if (!flag_s[0]) return;
  __threadfence();

  const size_t base = ((size_t)b * p.Hkv + kvh) * p.S;
  float* wts = reinterpret_cast<float*>(ring);  // [n_splits][GT]
  float* Ms = wts + kMaxSplits * GT;            // [GT]
  float* dens = Ms + GT;                        // [GT]
  for (int g = ctid; g < G; g += kConsumerThreads) {
    float M = -INFINITY;
    for (int s2 = 0; s2 < n_splits; ++s2) M = fmaxf(M, __ldcg(p.ws_m + (base + s2) * G + g));
    Ms[g] = M;
  }
  named_bar_sync(kMergeBar, kConsumerThreads);
  for (int i = ctid; i < n_splits * G; i += kConsumerThreads) {
    const int s2 = i / G, g = i - (i / G) * G;
    wts[s2 * GT + g] = exp2f(__ldcg(p.ws_m + (base + s2) * G + g) - Ms[g]);
  }
  named_bar_sync(kMergeBar, kConsumerThreads);
  for (int g = ctid; g < G; g += kConsumerThreads) {
    float den = 0.f;
    for (int s2 = 0; s2 < n_splits; ++s2) den += wts[s2 * GT + g] * __ldcg(p.ws_l + (base + s2) * G + g);
    dens[g] = den;
  }
  named_bar_sync(kMergeBar, kConsumerThreads);
  for (int i = ctid; i < G * D; i += kConsumerThreads) {
    const int g = i / D, d = i - (i / D) * D;
    float num = 0.f;
    for (int s2 = 0; s2 < n_splits; ++s2)
      num += wts[s2 * GT + g] * __ldcg(p.ws_acc + ((base + s2) * G + g) * D + d);
    out[(head0 + g) * D + d] = from_f32<T>(num / dens[g]);
  }
  if (ctid == 0) p.counters[(size_t)b * p.Hkv + kvh] = 0u;  // ready for the next call
}

// ------------------------------------------------------------------ launch
template <typename T, int D, int GT>
cudaError_t launch_decode_gt(const DecodeParams& p, cudaStream_t st) {
  using C = Cfg<D, GT>;
  // The dynamic shared memory opt-in is per device; remember which devices have it.
  static unsigned long long done_mask = 0ull;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(decode_kernel<T, D, GT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&done_mask, bit, __ATOMIC_ACQ_REL);
  }
  const dim3 grid(p.S, p.Hkv, p.B);
  decode_kernel<T, D, GT><<<grid, kThreads, C::SMEM, st>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_decode_dispatch(const DecodeParams& p, cudaStream_t st) {
  switch (p.G) {
    case 1: return launch_decode_gt<T, D, 1>(p, st);
    case 2: return launch_decode_gt<T, D, 2>(p, st);
    case 3: return launch_decode_gt<T, D, 3>(p, st);
    case 4: return launch_decode_gt<T, D, 4>(p, st);
    case 5: return launch_decode_gt<T, D, 5>(p, st);
    case 6: return launch_decode_gt<T, D, 6>(p, st);
    case 7: return launch_decode_gt<T, D, 7>(p, st);
    case 8: return launch_decode_gt<T, D, 8>(p, st);
    default: return launch_decode_gt<T, D, 16>(p, st);  // 9..16: padded heads are zero
  }
}

}  // namespace pa

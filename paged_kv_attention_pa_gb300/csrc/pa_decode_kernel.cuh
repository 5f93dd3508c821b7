// Split-KV single-query paged-attention decode for sm_103a.
//
// One CTA serves one (split, KV head, sequence): all G query heads of that KV
// head share every K/V tile it stages ("one workgroup per (sequence, KV head)"
// in "Hybrid-SSM decode rate on dual Radeon cards under vLLM", widened by the
// split-KV fix of the same page so that B * Hkv * splits fills every SM even at
// batch 1 with 4 KV heads).
//
// Loads. Every warp streams its own tiles of TW tokens (32 at head_dim 128 and
// for fp8 caches, 16 at head_dim 256) through a private ring of DEPTH shared-memory
// slots with 16-byte cp.async copies (L2 evict-first), DEPTH - 1 tiles in flight
// while it computes one: ~130-160 KB of loads in flight per SM. A warp's tiles are
// first those of its split's static share (tile j to warp j % NW), then tiles of
// the sequence's shared tail, claimed one at a time from a counter per (sequence,
// KV head), so that splits on faster SMs stream more of them. Only rows of live
// tokens (t < seq_len) are copied; the unwritten tail of the last block is never
// read ("vLLM's custom ROCm paged-attention kernel wins all sixty cells", §5,
// the V-load fault), and V rows past seq_len are zeroed (in shared memory, or in
// registers for fp8) so that the tensor-core sum over tokens only sees finite
// values there.
//
// Math. The GQA group's two contractions run on tensor cores per warp
// (mma.sync m16n8k16, fp32 accumulate), one MMA row block per 16 tokens:
// S^T[16 tokens x 8 heads] = K_tile q^T, then O^T[d x 8 heads] += V_tile^T P^T with
// P rounded to the MMA type. Scores of tokens past seq_len become -inf by select
// before the online softmax (exp2 domain, running max and sum per head). Groups
// of 9..16 heads (or query rows x heads) use two or four 8-column tiles. FP8 E4M3
// K and V bytes are widened exactly to fp16 in registers, straight into the MMA
// fragments.
//
// Epilogue: the warps merge their (m, l, acc) in shared memory. A sequence that
// fits in one split gets its output written here. Up to eight splits of a
// (sequence, KV head) can run as one thread-block cluster and merge through
// distributed shared memory. Otherwise the split's partial goes to the workspace
// and merge_kernel, chained behind this grid with a programmatic dependent launch,
// combines the splits of every (sequence, head) in parallel.
#pragma once

#include <cstdint>
#include <type_traits>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_params.h"

namespace pa {

constexpr int kSmemBudget = 224 * 1024;
#ifndef PA_CLUSTER_MERGE_MAX
#define PA_CLUSTER_MERGE_MAX 8  // largest split count merged in its cluster (2..8)
#endif

// F8: the cache holds FP8 E4M3 (one byte per element); tiles land in the ring as
// bytes, and each lane widens the bytes of its MMA fragments in registers.
template <int D, int NT, bool F8 = false>
struct Cfg {
  static constexpr int NW = warps_per_cta(D, F8);  // warps per CTA
  static constexpr int THREADS = NW * 32;
  static constexpr int TW = tile_tokens(D, F8);  // tokens per tile
  static_assert(TW % 16 == 0 && TW <= 32, "a tile is whole MMA row blocks, one token per lane");
  static constexpr int GT = 8 * NT;             // heads computed (G padded)
  static constexpr int KVB = F8 ? 1 : 2;        // bytes per cache element
  static constexpr int ROWB = D * KVB + 16;     // ring row pitch, padded against bank conflicts
  static constexpr int CPR = D * KVB / 16;      // 16-byte chunks per row
  static constexpr int TILE_BYTES = TW * ROWB;  // K (or V) half of a slot
  static constexpr int SLOT_BYTES = 2 * TILE_BYTES;
  static constexpr int KS = D / 16;             // k-steps of the score MMA = d-blocks of PV
  static constexpr int COPIES = TW * CPR / 32;  // 16-byte copies per lane per operand per tile
  static constexpr int FIXED = 256;
  static constexpr int DEPTH_FIT = (kSmemBudget - FIXED) / (NW * SLOT_BYTES);
  static constexpr int DEPTH = DEPTH_FIT > 12 ? 12 : DEPTH_FIT;  // slots per warp
  static constexpr int RING = NW * DEPTH * SLOT_BYTES;
  static constexpr int SMEM = RING + FIXED;
  static_assert((TW * CPR) % 32 == 0, "tile shape");
  static_assert(DEPTH >= 2, "need at least two slots per warp");
};

// t / block_size for a token index 0 <= t < 2^31 (see bs_magic)
__device__ __forceinline__ int div_block(const DecodeParams& p, int t) {
  return p.bs_magic == 0 ? (t >> p.bs_shift) : (int)(__umulhi((uint32_t)t, p.bs_magic) >> p.bs_shift);
}

// The cluster merge keeps, in the last warp's ring region after that warp's parked
// state, one receive entry of 12 floats (8 sums, maximum, denominator, padding) per
// split of the cluster and output item of this split's share: at most
// (items + splits) entries, items = 8 NT columns x D / 8.
constexpr int kRecvFloats = 12;
template <int D, int NT, bool F8>
__host__ __device__ constexpr bool cluster_merge_fits() {
  using C = Cfg<D, NT, F8>;
  return (8 * NT * (D + 6) + (8 * NT * (D / 8) + kMaxClusterMerge) * kRecvFloats) * 4 <=
         C::DEPTH * C::SLOT_BYTES;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(src), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// T: q and out type; KV: cache element type (T, or fp8e4m3 with fp16 MMAs).
template <typename T, typename KV, int D, int NT, bool WIN>
__global__ void __launch_bounds__(Cfg<D, NT, std::is_same_v<KV, fp8e4m3>>::THREADS, 1)
    decode_kernel(const DecodeParams p) {
  constexpr bool F8 = std::is_same_v<KV, fp8e4m3>;
  using TM = std::conditional_t<F8, __half, T>;  // MMA operand type
  using C = Cfg<D, NT, F8>;
  constexpr int GT = C::GT;
  constexpr int kWarps = C::NW;
  constexpr int kThreads = C::THREADS;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2;  // fragment row group
  const int tig = lane & 3;   // thread in group
  const int G = p.G;
  const int R = p.q_len;   // query rows per sequence (1 for single-query decode)
  const int cols = G * R;  // MMA columns: column c is (row c / G, head kvh*G + c % G)
  T* out = reinterpret_cast<T*>(p.out);
  auto qrow = [&](int c) -> size_t {  // row of q / out holding column c
    return ((size_t)b * R + c / G) * p.Hq + (size_t)kvh * G + c % G;
  };

  // Inputs may come from the previous kernel in the stream: wait for it (a no-op
  // without a programmatic launch). A split grid then lets its merge grid get
  // scheduled at once (small CTAs that prefetch the partials meanwhile); a grid
  // that writes the output itself lets the next kernel launch only once its CTAs
  // have streamed their tiles: the next call's CTAs, resident early on the SMs
  // this grid leaves idle, measured slower than a later launch.
  pdl_wait();
  if (p.S > 1 && !p.cmerge) pdl_launch_dependents();

  // ---- prologue: everything the first copies depend on is requested at once (one
  // round trip): the context length, the query fragments and, speculatively, the
  // block-table entries of this warp's first static tiles. Entries are read only
  // inside the table row; those past the sequence are ignored, never dereferenced.
  const int32_t* bt_row = p.block_tables + (size_t)b * p.max_blocks;
  const int cap = (int)min((long long)p.max_seq_len, (long long)p.max_blocks * p.block_size);
  int L = __ldg(p.seq_lens + b);
  auto validate_len = [&]() {
    if (L < 0 || L > cap) {
      if (split == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_SEQ_LEN);
      L = L < 0 ? 0 : cap;
    }
  };
  // A sliding window starts the context at max(0, L - window): its splits depend on
  // L, so only the full-context path requests the first table entries speculatively.
  int t_lo = 0;
  if constexpr (WIN) {
    validate_len();
    t_lo = max(0, L - p.window);
  }
  // This split owns Ps tokens from s_lo (its static share; Ps == P unless the
  // remaining tokens of the sequence are shared out tile by tile, see below).
  const int s_lo = t_lo + split * p.Ps;
  auto static_t0 = [&](int k) { return s_lo + (warp + k * kWarps) * C::TW; };
  // lanes 0..TW-1: block-table entry of token t0 + lane (0 where there is none)
  auto entry_of = [&](int t0) -> int {
    const long long t = (long long)t0 + lane;
    if (lane >= C::TW || t0 < 0 || t >= cap) return 0;
    return __ldg(bt_row + div_block(p, (int)t));
  };
  int pe[C::DEPTH];  // entries of tiles 0 .. DEPTH-1
#pragma unroll
  for (int k = 0; k < C::DEPTH; ++k) pe[k] = entry_of(static_t0(k));
  // query fragments (B operand of the score MMA), unscaled, zero for padded heads
  uint32_t qf[NT][C::KS][2];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = nt * 8 + gid;
      const bool ok = c < cols;
      const size_t rowp = (qrow(ok ? c : 0) * D) / 2;  // in bf16/f16 pairs
      if constexpr (F8) {
        // fp8 caches feed K to the MMA in a permuted d order: fragment elements
        // {2tig, 2tig+1, 2tig+8, 2tig+9} of k-step kk hold d = 4 KS tig + 4kk + {0..3},
        // so that a lane's K bytes of a row are contiguous; q takes the same order and
        // every dot product is unchanged. The lane's q words of the row are then
        // contiguous too (2 KS words from word 2 KS tig): 16-byte loads.
        const uint4* q4 = reinterpret_cast<const uint4*>(q32 + rowp) + (C::KS / 2) * tig;
#pragma unroll
        for (int j = 0; j < C::KS / 2; ++j) {
          const uint4 v = ok ? __ldg(q4 + j) : make_uint4(0u, 0u, 0u, 0u);
          qf[nt][2 * j][0] = v.x;
          qf[nt][2 * j][1] = v.y;
          qf[nt][2 * j + 1][0] = v.z;
          qf[nt][2 * j + 1][1] = v.w;
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < C::KS; ++kk) {
          qf[nt][kk][0] = ok ? __ldg(q32 + rowp + kk * 8 + tig) : 0u;
          qf[nt][kk][1] = ok ? __ldg(q32 + rowp + kk * 8 + 4 + tig) : 0u;
        }
      }
    }
  }

  // ---- context length, validated against the bounds the launch was planned for
  if constexpr (!WIN) validate_len();
  if (L == 0 && !p.cmerge) {  // empty context: zero rows, written once
    if (split == 0)
      for (int i = threadIdx.x; i < cols * D; i += kThreads)
        out[qrow(i / D) * D + i % D] = from_f32<T>(0.f);
    return;
  }
  // a split past the sequence has nothing to do (in a merging cluster it streams
  // nothing and still meets its partner at the cluster barriers)
  const bool past = t_lo + split * p.P >= L;
  if (past && !p.cmerge) return;
  const int n_splits = (L - t_lo + p.P - 1) / p.P;
  // Work sharing among the splits of one (sequence, KV head). Every split streams
  // its static share; the tokens past the n static shares go out one tile at a
  // time from a counter in the workspace, so that splits on faster SMs take more of
  // them and all end together. The merge kernel resets the counter.
  const bool steal = p.Ps < p.P && n_splits > 1;
  const int s_hi = steal ? min(L, s_lo + p.Ps) : min(L, t_lo + (split + 1) * p.P);
  // static tiles of the CTA (>= 1 unless past the sequence: its s_lo counts static
  // shares, which may start inside the context that the first split covers alone)
  const int n_stat = past ? 0 : (s_hi - s_lo + C::TW - 1) / C::TW;
  const int ns = warp < n_stat ? (n_stat - warp + kWarps - 1) / kWarps : 0;  // this warp's
  const int dyn_lo = steal ? min(L, t_lo + n_splits * p.Ps) : L;
  const int n_dyn = (L - dyn_lo + C::TW - 1) / C::TW;  // shared tiles of the sequence
  int* const ctr = steal ? p.steal + (size_t)b * p.Hkv + kvh : nullptr;
  // Causal limit of each of this thread's columns: row i sees tokens t < L - R + i + 1
  // (all of them when R = 1).
  int lim[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) lim[nt][h] = L - R + (nt * 8 + 2 * tig + h) / G + 1;

  // ---- per-warp copy pipeline
  const uint64_t pol = l2_evict_first_policy();
  const uint8_t* kbase = reinterpret_cast<const uint8_t*>(p.k_cache);
  const ptrdiff_t v_minus_k =
      reinterpret_cast<const uint8_t*>(p.v_cache) - reinterpret_cast<const uint8_t*>(p.k_cache);
  uint8_t* my_ring = ring + warp * C::DEPTH * C::SLOT_BYTES;
  const uint32_t my_ring_s = smem_addr(my_ring);

  // Issue the copies of this warp's k-th tile, tokens t0 .. (a commit group even
  // when t0 < 0: no tile); phys is this lane's block-table entry, validated here.
  auto issue = [&](int k, int phys, int t0) {
    if (t0 >= 0) {
      const int nv = min(C::TW, L - t0);
      // lanes 0..TW-1 resolve one row each: cache row index of token t0 + lane
      uint32_t ridx = 0;
      if (lane < nv) {
        const int t = t0 + lane;
        const int off = t - div_block(p, t) * p.block_size;
        if ((unsigned)phys >= (unsigned)p.num_blocks) {
          atomicOr(p.err, PA_DEVERR_BLOCK_INDEX);
          phys = 0;
        }
        ridx = ((uint32_t)phys * (uint32_t)p.block_size + (uint32_t)off) * (uint32_t)p.Hkv +
               (uint32_t)kvh;
      }
      const uint32_t slot = my_ring_s + (k % C::DEPTH) * C::SLOT_BYTES;
#pragma unroll
      for (int i = 0; i < C::COPIES; ++i) {
        const int flat = i * 32 + lane;
        const int r = flat / C::CPR, c = flat % C::CPR;
        const uint32_t rr = __shfl_sync(0xffffffffu, ridx, r);
        if (r < nv) {
          const uint8_t* src = kbase + (size_t)rr * (D * C::KVB) + c * 16;
          const uint32_t dst = slot + r * C::ROWB + c * 16;
          cp_async16(dst, src, pol);
          cp_async16(dst + C::TILE_BYTES, src + v_minus_k, pol);
        }
      }
    }
    cp_async_commit();
  };

  // This warp's tiles: its static ones, then shared ones. A shared tile is claimed
  // one step before its block-table entry is requested (lane 0's atomic, still in
  // flight meanwhile). The stream ends at the first claim past the shared tiles,
  // so no claim is left unconsumed.
  int kk_next = 0;        // index of the next tile to define
  int claim = 0;          // lane 0: result of the claim in flight
  bool claiming = false;  // a claim is in flight
  bool more = n_dyn > 0;  // shared tiles may remain
  auto next_t0 = [&]() -> int {  // t0 of the next tile of the stream, -1 past its end
    const int kk = kk_next++;
    int t0 = -1;
    if (kk < ns) {
      t0 = static_t0(kk);
    } else if (more) {
      if (!claiming && lane == 0) claim = atomicAdd(ctr, 1);
      const int g = __shfl_sync(0xffffffffu, claim, 0);
      claiming = false;
      if (g < n_dyn)
        t0 = dyn_lo + g * C::TW;
      else
        more = false;
    }
    if (more && !claiming && kk + 1 >= ns) {  // claim the tile after this one now
      if (lane == 0) claim = atomicAdd(ctr, 1);
      claiming = true;
    }
    return t0;
  };
  // The first DEPTH tiles: the static ones among the first DEPTH - 1 go out at
  // once; the shared ones are claimed together (one atomic) and go out when their
  // entries arrive; then the claim of tile DEPTH goes out.
#pragma unroll
  for (int k = 0; k < C::DEPTH - 1; ++k)
    if (k < ns) issue(k, pe[k], static_t0(k));
  int tq[C::DEPTH];  // t0 of tiles k .. k + DEPTH - 1
  {
    const int m0 = ns < C::DEPTH ? C::DEPTH - ns : 0;
    int g0 = 0;
    if (m0 > 0 && more) {
      if (lane == 0) g0 = atomicAdd(ctr, m0);
      g0 = __shfl_sync(0xffffffffu, g0, 0);
    }
#pragma unroll
    for (int k = 0; k < C::DEPTH; ++k) {
      if (k < ns) {
        tq[k] = static_t0(k);
      } else {
        const int g = g0 + (k - ns);
        if (more && g >= n_dyn) more = false;
        tq[k] = more ? dyn_lo + g * C::TW : -1;
        pe[k] = entry_of(tq[k]);  // not a static tile: look its entry up now
      }
    }
    kk_next = C::DEPTH;
    if (more && ns <= C::DEPTH) {
      if (lane == 0) claim = atomicAdd(ctr, 1);
      claiming = true;
    }
  }

#pragma unroll
  for (int k = 0; k < C::DEPTH - 1; ++k)
    if (k >= ns) issue(k, pe[k], tq[k]);
  int next_entry = pe[C::DEPTH - 1];  // for the tile issued in the first loop iteration
  if constexpr (F8 && !std::is_same_v<T, __half>) {
    // bf16 queries as fp16 pairs for the fp8 path's fp16 MMAs. Converted only now:
    // done in the prologue, the conversion made the warp wait for the query's round
    // trip before it could issue its first copies.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int kk = 0; kk < C::KS; ++kk) {
        const float2 a0 = unpack2<T>(qf[nt][kk][0]), a1 = unpack2<T>(qf[nt][kk][1]);
        qf[nt][kk][0] = pack2<__half>(a0.x, a0.y);
        qf[nt][kk][1] = pack2<__half>(a1.x, a1.y);
      }
  }

  // running state: this thread's heads are nt*8 + 2*tig + {0, 1}
  float m[NT][2], l[NT][2];
  float o[NT][C::KS][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = -INFINITY;
    l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
    for (int dd = 0; dd < C::KS; ++dd) o[nt][dd][0] = o[nt][dd][1] = o[nt][dd][2] = o[nt][dd][3] = 0.f;
  }
  // ldmatrix row addresses (byte offsets inside a 16-bit tile) for this lane
  const uint32_t k_lane = (uint32_t)(((lane & 7) + 8 * ((lane >> 3) & 1)) * C::ROWB + (lane >> 4) * 16);
  const uint32_t v_lane = (uint32_t)(((lane & 7) + 8 * (lane >> 4)) * C::ROWB + ((lane >> 3) & 1) * 16);
  const float sl2 = p.scale_log2;
  constexpr bool kLazy = F8;                 // see the rescaling in the softmax
  constexpr float kSlack = kLazy ? 8.f : 0.f;  // log2 units

  for (int k = 0; tq[0] >= 0; ++k) {  // tile k of the stream: tokens tq[0] ..
    const int entry = next_entry;
    const int t_new = next_t0();    // tile k + DEPTH
    next_entry = entry_of(t_new);   // one iteration ahead of its use
    issue(k + C::DEPTH - 1, entry, tq[C::DEPTH - 1]);
    cp_async_wait<C::DEPTH - 1>();  // tile k has landed (for this lane's copies)
    const int t0 = tq[0];
#pragma unroll
    for (int i = 0; i + 1 < C::DEPTH; ++i) tq[i] = tq[i + 1];
    tq[C::DEPTH - 1] = t_new;
    const int nv = min(C::TW, L - t0);
    const uint32_t kt = my_ring_s + (k % C::DEPTH) * C::SLOT_BYTES;
    const uint32_t vt = kt + C::TILE_BYTES;
    if constexpr (!F8) {
      if (nv < C::TW) {
        // rows past seq_len were never loaded: zero them in V so that p = 0 meets 0
        uint8_t* vrow = my_ring + (k % C::DEPTH) * C::SLOT_BYTES + C::TILE_BYTES;
        for (int i = lane; i < (C::TW - nv) * C::CPR; i += 32) {
          const int r = nv + i / C::CPR, c = i % C::CPR;
          *reinterpret_cast<uint4*>(vrow + r * C::ROWB + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    __syncwarp();  // every lane's copies (and the zero rows) are visible

    // ---- scores S^T[token][head] = K_tile . q^T (fp32 accumulate), one MMA row
    // block per 16 tokens (mt); two independent accumulator chains (even / odd
    // k-steps) halve the MMA latency
    constexpr int MT = C::TW / 16;
    float s[MT][NT][4], s2[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[mt][nt][i] = s2[mt][nt][i] = 0.f;
    // fp8: this lane's K bytes d in [4 KS tig, 4 KS tig + 4 KS) of rows 16mt + gid and
    // 16mt + gid + 8 (rows past seq_len hold stale bytes: their scores become -inf)
    uint4 kw[MT][2][F8 ? C::KS / 4 : 1];
    if constexpr (F8) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int u = 0; u < C::KS / 4; ++u) {
          kw[mt][0][u] = lds128(kt + (16 * mt + gid) * C::ROWB + 4 * C::KS * tig + 16 * u);
          kw[mt][1][u] = lds128(kt + (16 * mt + gid + 8) * C::ROWB + 4 * C::KS * tig + 16 * u);
        }
    }
#pragma unroll
    for (int kk = 0; kk < C::KS; ++kk) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t a[4];
        if constexpr (F8) {
          // k-step kk: d = 4 KS tig + 4kk .. +3 of the two rows
          const uint32_t w0 = word_of(kw[mt][0][kk / 4], kk % 4);
          const uint32_t w1 = word_of(kw[mt][1][kk / 4], kk % 4);
          a[0] = e4m3x2_to_half2(w0 & 0xffff);
          a[2] = e4m3x2_to_half2(w0 >> 16);
          a[1] = e4m3x2_to_half2(w1 & 0xffff);
          a[3] = e4m3x2_to_half2(w1 >> 16);
        } else {
          ldmatrix_x4<false>(a, kt + 16 * mt * C::ROWB + k_lane + kk * 32);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (kk & 1)
            mma16816<TM>(s2[mt][nt], a, qf[nt][kk][0], qf[nt][kk][1]);
          else
            mma16816<TM>(s[mt][nt], a, qf[nt][kk][0], qf[nt][kk][1]);
        }
      }
    }
    // ---- online softmax over the tile. Tokens 16mt + gid (+ 8); -inf by select past
    // each column's limit (seq_len, and the causal limit of the column's query row);
    // rows past seq_len were never loaded
    uint32_t pb[MT][NT][2];
    float x[NT][MT][4];
    float mx[NT][2];
    bool grow = false;  // some column of this lane sees a score above its running max (+ slack)
    if (t0 + C::TW <= L - R + 1) {
      // every token of the tile is below every column's limit (the usual case): no mask
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) x[nt][mt][i] = (s[mt][nt][i] + s2[mt][nt][i]) * sl2;
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int tok0 = t0 + 16 * mt + gid, tok1 = tok0 + 8;
          x[nt][mt][0] = tok0 < lim[nt][0] ? (s[mt][nt][0] + s2[mt][nt][0]) * sl2 : -INFINITY;
          x[nt][mt][1] = tok0 < lim[nt][1] ? (s[mt][nt][1] + s2[mt][nt][1]) * sl2 : -INFINITY;
          x[nt][mt][2] = tok1 < lim[nt][0] ? (s[mt][nt][2] + s2[mt][nt][2]) * sl2 : -INFINITY;
          x[nt][mt][3] = tok1 < lim[nt][1] ? (s[mt][nt][3] + s2[mt][nt][3]) * sl2 : -INFINITY;
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mx[nt][0] = mx[nt][1] = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mx[nt][0] = fmaxf(mx[nt][0], fmaxf(x[nt][mt][0], x[nt][mt][2]));
        mx[nt][1] = fmaxf(mx[nt][1], fmaxf(x[nt][mt][1], x[nt][mt][3]));
      }
      grow = grow || mx[nt][0] > m[nt][0] + kSlack || mx[nt][1] > m[nt][1] + kSlack;
    }
    // 16-bit caches: most tiles raise no running max (all scale factors are exactly
    // 1) and skip the cross-lane maxima and the rescaling, with bit-identical
    // results; at head_dim 256, and with more than 8 columns, the skip measured
    // slower per call: every tile rescales there.
    // FP8 caches (bound by instruction issue): the running max is a reference point,
    // not necessarily the maximum. Weights are 2^(s - m) against the m in use and the
    // sums and accumulators stay relative to the same m, so any m gives the same
    // softmax; m is raised only when a score exceeds it by more than kSlack (weights
    // stay <= 2^kSlack, exact in fp32 and rounded like any weight to fp16), so
    // almost every tile skips the rescaling.
    const bool rescale = (!kLazy && (D != 128 || NT > 1)) || __any_sync(0xffffffffu, grow);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float al0 = 1.f, al1 = 1.f;
      if (rescale) {
        float mx0 = mx[nt][0], mx1 = mx[nt][1];
        // tile max per head over its tokens (lanes sharing tig)
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
        }
        const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
        const float q0 = mn0 == -INFINITY ? 0.f : mn0, q1 = mn1 == -INFINITY ? 0.f : mn1;
        al0 = exp2_approx(m[nt][0] - q0);
        al1 = exp2_approx(m[nt][1] - q1);
        m[nt][0] = mn0;
        m[nt][1] = mn1;
#pragma unroll
        for (int dd = 0; dd < C::KS; ++dd) {
          o[nt][dd][0] *= al0;
          o[nt][dd][1] *= al1;
          o[nt][dd][2] *= al0;
          o[nt][dd][3] *= al1;
        }
      }
      const float r0 = m[nt][0] == -INFINITY ? 0.f : m[nt][0];
      const float r1 = m[nt][1] == -INFINITY ? 0.f : m[nt][1];
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const float p0 = exp2_approx(x[nt][mt][0] - r0), p1 = exp2_approx(x[nt][mt][1] - r1);
        const float p2 = exp2_approx(x[nt][mt][2] - r0), p3 = exp2_approx(x[nt][mt][3] - r1);
        ps0 += p0 + p2;
        ps1 += p1 + p3;
        // P^T[token][head] fragments -> P[head][token] as the B operand of PV
        pb[mt][nt][0] = movmatrix_trans(pack2<TM>(p0, p1));
        pb[mt][nt][1] = movmatrix_trans(pack2<TM>(p2, p3));
      }
      l[nt][0] = l[nt][0] * al0 + ps0;
      l[nt][1] = l[nt][1] * al1 + ps1;
    }

    // ---- O^T[d][head] += V_tile^T . P^T, one MMA per d-block and row block
    if constexpr (F8) {
      // Rows of the V^T fragments are permuted: in d-block dd, row gid holds
      // d = 2 KS gid + 2dd and row gid + 8 holds d + 1, so that a lane needs bytes
      // [2 KS gid, 2 KS gid + 2 KS) of its tokens 16mt + {2tig, 2tig+1, 2tig+8,
      // 2tig+9}: one or two 16-byte loads per token, then a byte permute pairs two
      // tokens of one d for each fp16x2 register. Rows past seq_len read as 0.
      uint4 vw[MT][4][C::KS / 8];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 16 * mt + 2 * tig + (j & 1) + 8 * (j >> 1);
#pragma unroll
          for (int u = 0; u < C::KS / 8; ++u) vw[mt][j][u] = lds128(vt + r * C::ROWB + 2 * C::KS * gid + 16 * u);
        }
      if (nv < C::TW) {  // a partial tile: its rows past seq_len were never loaded
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 16 * mt + 2 * tig + (j & 1) + 8 * (j >> 1);
#pragma unroll
            for (int u = 0; u < C::KS / 8; ++u)
              if (r >= nv) vw[mt][j][u] = make_uint4(0u, 0u, 0u, 0u);
          }
      }
#pragma unroll
      for (int dd = 0; dd < C::KS; ++dd) {
        const int wi = dd >> 1;                             // word of bytes 2dd, 2dd + 1
        const uint32_t sel = (dd & 1) ? 0x7362u : 0x5140u;  // pair bytes 2,3 or 0,1
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t p01 = __byte_perm(word_of(vw[mt][0][wi / 4], wi % 4),
                                           word_of(vw[mt][1][wi / 4], wi % 4), sel);
          const uint32_t p23 = __byte_perm(word_of(vw[mt][2][wi / 4], wi % 4),
                                           word_of(vw[mt][3][wi / 4], wi % 4), sel);
          uint32_t a[4];
          a[0] = e4m3x2_to_half2(p01 & 0xffff);  // row gid:     tokens 2tig, 2tig+1
          a[1] = e4m3x2_to_half2(p01 >> 16);     // row gid + 8: tokens 2tig, 2tig+1
          a[2] = e4m3x2_to_half2(p23 & 0xffff);  // row gid:     tokens 2tig+8, 2tig+9
          a[3] = e4m3x2_to_half2(p23 >> 16);     // row gid + 8: tokens 2tig+8, 2tig+9
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816<TM>(o[nt][dd], a, pb[mt][nt][0], pb[mt][nt][1]);
        }
      }
    } else {
#pragma unroll
      for (int dd = 0; dd < C::KS; ++dd) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a[4];
          ldmatrix_x4<true>(a, vt + 16 * mt * C::ROWB + v_lane + dd * 32);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816<TM>(o[nt][dd], a, pb[mt][nt][0], pb[mt][nt][1]);
        }
      }
    }
    __syncwarp();  // every lane is done with this slot before it is refilled
  }
  cp_async_wait<0>();

  if (p.S == 1 || p.cmerge) pdl_launch_dependents();

  // ---- denominators: sum over the 8 lanes that share tig (different tokens)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) l[nt][h] += __shfl_xor_sync(0xffffffffu, l[nt][h], o2);

  // ---- merge the warps. Each warp writes its state (m, l, unscaled accumulators)
  // into its own ring, which only it has used: every one of its copies has landed
  // and been consumed. After one barrier, the final pass reads all warps' states
  // and weighs each by 2^(m_w - M) with M the CTA maximum of the column: it sums
  // 8 consecutive d of one column per item as two 16-byte words per warp and
  // writes them with one 16-byte store. Accumulator rows are padded by 4 floats,
  // so that the fragment writes (columns 2 tig + {0, 1}, rows gid) fall in
  // distinct banks.
  constexpr int AP = D + 4;
  constexpr int WSTATE = GT * (AP + 2);  // floats of one warp's state
  static_assert(WSTATE * 4 <= C::DEPTH * C::SLOT_BYTES, "a warp's state fits in its ring");
  auto wstate = [&](int w) { return reinterpret_cast<float*>(ring + w * C::DEPTH * C::SLOT_BYTES); };
  {
    float* mw = wstate(warp);  // [GT] running maxima, [GT] sums, [GT][AP] accumulators
    float* lw = mw + GT;
    float* aw = lw + GT;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c0 = nt * 8 + 2 * tig;
      if (gid == 0) {
        mw[c0] = m[nt][0];
        mw[c0 + 1] = m[nt][1];
        lw[c0] = l[nt][0];
        lw[c0 + 1] = l[nt][1];
      }
      float* a0 = aw + c0 * AP;
#pragma unroll
      for (int dd = 0; dd < C::KS; ++dd) {
        // rows gid and gid + 8 of d-block dd (permuted for fp8 caches, see the PV step)
        const int dlo = F8 ? 2 * C::KS * gid + 2 * dd : dd * 16 + gid;
        const int dhi = F8 ? dlo + 1 : dlo + 8;
        a0[dlo] = o[nt][dd][0];
        a0[AP + dlo] = o[nt][dd][1];
        a0[dhi] = o[nt][dd][2];
        a0[AP + dhi] = o[nt][dd][3];
      }
    }
  }
  __syncthreads();

  const bool single = n_splits == 1;
  const size_t pidx = ((size_t)b * p.Hkv + kvh) * p.S + split;
  constexpr int DV = D / 8;  // items per column
  // The cluster merge: the C = p.cmerge splits of this (sequence, KV head) form one
  // cluster. Split r owns output items [r per, (r + 1) per); every split pushes its
  // state of each item into the owner's receive entries (distributed shared memory
  // stores, which need no round trip), and after a cluster barrier every owner
  // reduces its items from its own shared memory.
  const int ccount = p.cmerge;
  const int cper = ccount ? (cols * DV + ccount - 1) / ccount : 0;
  float* const recv = wstate(kWarps - 1) + WSTATE;  // [C][cper][kRecvFloats]
  if constexpr (cluster_merge_fits<D, NT, F8>()) {
    // every split of the cluster is past its main loop: the receive entries (in ring
    // memory) are free
    if (ccount) cluster_sync_relaxed();  // orders execution: nothing is pending on them
  }
  for (int it = threadIdx.x; it < cols * DV; it += kThreads) {
    const int g = it / DV, d0 = (it % DV) * 8;  // g: column
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wstate(w)[g]);
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* st = wstate(w);
      const float mwg = st[g];
      // a warp that saw no token of the column (m = -inf) contributes nothing
      const float f = mwg == -INFINITY ? 0.f : exp2_approx(mwg - M);
      const float4* src = reinterpret_cast<const float4*>(st + 2 * GT + g * AP + d0);
      const float4 x = src[0], y = src[1];
      v[0] += f * x.x; v[1] += f * x.y; v[2] += f * x.z; v[3] += f * x.w;
      v[4] += f * y.x; v[5] += f * y.y; v[6] += f * y.z; v[7] += f * y.w;
      den += f * st[GT + g];
    }
    // cache values are stored values times v_scale (1 unless fp8); a column whose
    // row sees no token of this split has M = -inf and den = 0
    if constexpr (cluster_merge_fits<D, NT, F8>()) {
      if (ccount) {  // this split's state of the item, pushed to the item's owner
        const int owner = it / cper;
        float* e = const_cast<float*>(map_cluster_rank(recv, (uint32_t)owner)) +
                   ((size_t)cluster_rank() * cper + (it - owner * cper)) * kRecvFloats;
        reinterpret_cast<float4*>(e)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(e)[1] = make_float4(v[4], v[5], v[6], v[7]);
        reinterpret_cast<float2*>(e)[4] = make_float2(M, den);
        continue;
      }
    }
    if (single) {
      const float r = den > 0.f ? p.v_scale / den : 0.f;
      uint4 pk;
      pk.x = pack2<T>(v[0] * r, v[1] * r);
      pk.y = pack2<T>(v[2] * r, v[3] * r);
      pk.z = pack2<T>(v[4] * r, v[5] * r);
      pk.w = pack2<T>(v[6] * r, v[7] * r);
      *reinterpret_cast<uint4*>(out + qrow(g) * D + d0) = pk;
    } else {
      const float vs = p.v_scale;
      float4* dst = reinterpret_cast<float4*>(p.ws_acc + (pidx * cols + g) * D + d0);
      dst[0] = make_float4(v[0] * vs, v[1] * vs, v[2] * vs, v[3] * vs);
      dst[1] = make_float4(v[4] * vs, v[5] * vs, v[6] * vs, v[7] * vs);
      if (d0 == 0) {
        p.ws_m[pidx * cols + g] = M;
        p.ws_l[pidx * cols + g] = den;
      }
    }
  }
  if constexpr (cluster_merge_fits<D, NT, F8>()) {
    if (ccount) {
      cluster_sync();  // every push has landed; no split reads another's memory after this
      const int rank = (int)cluster_rank();
      if (rank == 0 && p.Ps < p.P && threadIdx.x == 0)
        p.steal[(size_t)b * p.Hkv + kvh] = 0;  // no claims left
      const int i_lo = rank * cper, i_hi = min(cols * DV, i_lo + cper);
      for (int it = i_lo + threadIdx.x; it < i_hi; it += kThreads) {
        const int g = it / DV, d0 = (it % DV) * 8;
        const float* e0 = recv + (size_t)(it - i_lo) * kRecvFloats;
        // every entry loaded first, then the reduction
        float2 ml[kMaxClusterMerge];
        float4 xc[kMaxClusterMerge], yc[kMaxClusterMerge];
        float M = -INFINITY;
#pragma unroll
        for (int c2 = 0; c2 < kMaxClusterMerge; ++c2) {
          if (c2 < ccount) {
            const float* e = e0 + (size_t)c2 * cper * kRecvFloats;
            xc[c2] = reinterpret_cast<const float4*>(e)[0];
            yc[c2] = reinterpret_cast<const float4*>(e)[1];
            ml[c2] = reinterpret_cast<const float2*>(e)[4];
            M = fmaxf(M, ml[c2].x);
          }
        }
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float den = 0.f;
#pragma unroll
        for (int c2 = 0; c2 < kMaxClusterMerge; ++c2) {
          if (c2 < ccount) {
            // a split that saw no token of the column (m = -inf) weighs 0
            const float w = ml[c2].x == -INFINITY ? 0.f : exp2_approx(ml[c2].x - M);
            const float4 x = xc[c2], y = yc[c2];
            den += w * ml[c2].y;
            v[0] += w * x.x; v[1] += w * x.y; v[2] += w * x.z; v[3] += w * x.w;
            v[4] += w * y.x; v[5] += w * y.y; v[6] += w * y.z; v[7] += w * y.w;
          }
        }
        const float r = den > 0.f ? p.v_scale / den : 0.f;
        uint4 pk;
        pk.x = pack2<T>(v[0] * r, v[1] * r);
        pk.y = pack2<T>(v[2] * r, v[3] * r);
        pk.z = pack2<T>(v[4] * r, v[5] * r);
        pk.w = pack2<T>(v[6] * r, v[7] * r);
        *reinterpret_cast<uint4*>(out + qrow(g) * D + d0) = pk;
      }
    }
  }
}

// Combine the split partials of one (sequence, query head, 64-wide slice of D):
//   M = max_s m_s,  w_s = 2^(m_s - M),  out = sum_s w_s acc_s / sum_s w_s l_s
// (the flash-decoding reduction). Splits where a row sees no token carry m = -inf
// and weight 0. M is finite whenever the row sees a token; a row that sees none
// (several query rows, short context) is written as zeros. 256 threads: 64 output
// elements x 4 split lanes. Every warp reduces the maxima and sums itself with
// shuffles (lane s % 32 holds split s), so one barrier remains: the sum over the
// four split lanes.
template <typename T, int D>
__global__ void __launch_bounds__(256) merge_kernel(const DecodeParams p) {
  constexpr int kPre = 16, kReg = 2;  // 4 * kPre == 32 * kReg
  __shared__ float part[4][64];
  const int b = blockIdx.z, row = blockIdx.y / p.Hq, h = blockIdx.y % p.Hq;
  const int G = p.G, kvh = h / G, g = h - kvh * G;
  const int cols = G * p.q_len, c = row * G + g;  // the partials' column of (row, head)
  const size_t base = ((size_t)b * p.Hkv + kvh) * p.S;
  const int tid = threadIdx.x, lane = tid & 31;
  const int dl = tid & 63, sl = tid >> 6;
  const int d = blockIdx.x * 64 + dl;
  const float* acc = p.ws_acc + (base * cols + c) * D + d;
  const float* pm = p.ws_m + base * cols + c;
  const float* pl = p.ws_l + base * cols + c;
  // This grid starts while the decode grid finishes. Before waiting for it, ask for
  // the lines (and address translations) of this CTA's partials in L2, where the
  // decode grid writes them: a prefetch returns nothing, so it cannot read stale data.
  if (lane == 0)
    for (int i = 0; i < kPre; ++i)
      if (sl + 4 * i < p.S) prefetch_l2(acc + (size_t)(sl + 4 * i) * cols * D);
  if (tid < 32 * kReg && tid < p.S) {
    prefetch_l2(pm + (size_t)tid * cols);
    prefetch_l2(pl + (size_t)tid * cols);
  }
  pdl_wait();  // the partials of the decode grid are complete and visible
  pdl_launch_dependents();
  // One round trip: the context length, this thread's accumulators of splits sl + 4 i
  // (i < 16) and the warp's maxima and sums of splits lane and lane + 32, all within
  // the S splits launched. Splits past this sequence's own count wrote nothing: their
  // slots hold stale values, replaced by select once the count is known.
  float av[kPre];
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int s2 = sl + 4 * i;
    av[i] = s2 < p.S ? __ldcg(acc + (size_t)s2 * cols * D) : 0.f;
  }
  float mr[kReg], lr[kReg];
#pragma unroll
  for (int j = 0; j < kReg; ++j) {
    const int s2 = lane + 32 * j;
    mr[j] = s2 < p.S ? __ldcg(pm + (size_t)s2 * cols) : -INFINITY;
    lr[j] = s2 < p.S ? __ldcg(pl + (size_t)s2 * cols) : 0.f;
  }
  int L = __ldg(p.seq_lens + b);
  const int cap = (int)min((long long)p.max_seq_len, (long long)p.max_blocks * p.block_size);
  L = L < 0 ? 0 : (L > cap ? cap : L);
  if (p.window > 0) L = min(L, p.window);  // tokens the splits cover
  const int n = (L + p.P - 1) / p.P;
  if (n <= 1) return;  // written by the decode grid
  // the decode grid is done with this (sequence, KV head)'s tile counter: rearm it
  if (p.Ps < p.P && blockIdx.x == 0 && row == 0 && g == 0 && threadIdx.x == 0)
    p.steal[(size_t)b * p.Hkv + kvh] = 0;
#pragma unroll
  for (int i = 0; i < kPre; ++i) av[i] = sl + 4 * i < n ? av[i] : 0.f;
#pragma unroll
  for (int j = 0; j < kReg; ++j) {
    const bool live = lane + 32 * j < n;
    mr[j] = live ? mr[j] : -INFINITY;
    lr[j] = live ? lr[j] : 0.f;
  }
  float M = fmaxf(mr[0], mr[1]);
  for (int s2 = lane + 32 * kReg; s2 < n; s2 += 32) M = fmaxf(M, __ldcg(pm + (size_t)s2 * cols));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float wr[kReg], den = 0.f;
#pragma unroll
  for (int j = 0; j < kReg; ++j) {
    wr[j] = M == -INFINITY ? 0.f : exp2_approx(mr[j] - M);
    den += wr[j] * lr[j];
  }
  for (int s2 = lane + 32 * kReg; s2 < n; s2 += 32)
    den += M == -INFINITY ? 0.f : exp2_approx(__ldcg(pm + (size_t)s2 * cols) - M) * __ldcg(pl + (size_t)s2 * cols);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);

  float num = 0.f;
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int s2 = sl + 4 * i;  // held by lane s2 % 32 in wr[s2 / 32] (s2 / 32 == i / 8)
    num += __shfl_sync(0xffffffffu, wr[i / 8], s2 & 31) * av[i];
  }
  for (int s2 = sl + 4 * kPre; s2 < n; s2 += 4)
    num += M == -INFINITY ? 0.f : exp2_approx(__ldcg(pm + (size_t)s2 * cols) - M) * __ldcg(acc + (size_t)s2 * cols * D);
  part[sl][dl] = num;
  __syncthreads();
  if (sl == 0) {
    num = part[0][dl] + part[1][dl] + part[2][dl] + part[3][dl];
    reinterpret_cast<T*>(p.out)[(((size_t)b * p.q_len + row) * p.Hq + h) * D + d] =
        from_f32<T>(den > 0.f ? num / den : 0.f);
  }
}

// ------------------------------------------------------------------ launch
// Launch with programmatic stream serialization: the grid may start while the
// previous kernel in the stream finishes; its pdl_wait() orders the reads.
// cluster_x > 1 groups that many consecutive CTAs along x into a thread-block cluster.
template <typename Kern>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       const DecodeParams& p, unsigned cluster_x = 1) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename T, typename KV, int D, int NT, bool WIN>
cudaError_t launch_decode_nt(const DecodeParams& p, cudaStream_t st, int* kernels) {
  using C = Cfg<D, NT, std::is_same_v<KV, fp8e4m3>>;
  auto kern = decode_kernel<T, KV, D, NT, WIN>;
  // The dynamic shared memory opt-in is per device; remember which devices have it.
  static unsigned long long done_mask = 0ull;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&done_mask, bit, __ATOMIC_ACQ_REL);
  }
  DecodeParams q = p;
  // The splits of each (sequence, KV head) merge inside their cluster (no merge grid)
  // when their states fit: always for two splits; for three to kMaxClusterMerge when
  // every cluster of the launch is resident at once (clusters of more than two CTAs
  // pack the SMs less densely, so a launch of several waves keeps the merge grid).
  q.cmerge = 0;
  if (cluster_merge_fits<D, NT, std::is_same_v<KV, fp8e4m3>>() && q.S >= 2 &&
      q.S <= PA_CLUSTER_MERGE_MAX && q.S <= kMaxClusterMerge) {
    if (q.S == 2) {
      q.cmerge = 2;
    } else if (dev < 64) {
      static int clusters[64][kMaxClusterMerge + 1] = {};  // resident clusters, per size
      int n = __atomic_load_n(&clusters[dev][q.S], __ATOMIC_ACQUIRE);
      if (n == 0) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(q.S, q.Hkv, q.B);
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = q.S;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int got = 0;
        if (cudaOccupancyMaxActiveClusters(&got, kern, &cfg) != cudaSuccess) {
          cudaGetLastError();
          got = 0;
        }
        n = got > 0 ? got : -1;
        __atomic_store_n(&clusters[dev][q.S], n, __ATOMIC_RELEASE);
      }
      if (n > 0 && (long long)q.B * q.Hkv <= n) q.cmerge = q.S;
    }
  }
  if (kernels) {  // the count only
    *kernels = (q.S > 1 && !q.cmerge) ? 2 : 1;
    return cudaSuccess;
  }
  e = launch_pdl(kern, dim3(q.S, q.Hkv, q.B), dim3(C::THREADS), C::SMEM, st, q,
                 q.cmerge ? (unsigned)q.cmerge : 1u);
  if (e != cudaSuccess) return e;
  if (q.S > 1 && !q.cmerge)
    e = launch_pdl(merge_kernel<T, D>, dim3(D / 64, q.Hq * q.q_len, q.B), dim3(256), 0, st, q);
  return e;
}

// Column tiles of 8: one for up to 8 (row, head) columns, two for 16, four for 32
// (head_dim 128 only, no window: the host rejects the rest).
template <typename T, typename KV, int D>
cudaError_t launch_decode_dispatch(const DecodeParams& p, cudaStream_t st, int* kernels) {
  const int cols = p.G * p.q_len;
  if (p.window > 0)
    return cols <= 8 ? launch_decode_nt<T, KV, D, 1, true>(p, st, kernels)
                     : launch_decode_nt<T, KV, D, 2, true>(p, st, kernels);
  if (cols <= 8) return launch_decode_nt<T, KV, D, 1, false>(p, st, kernels);
  if (cols <= 16 || D != 128) return launch_decode_nt<T, KV, D, 2, false>(p, st, kernels);
  if constexpr (D == 128) return launch_decode_nt<T, KV, D, 4, false>(p, st, kernels);
  return cudaErrorInvalidValue;
}

}  // namespace pa

// Host side of libpa.so: argument validation, the split plan, the workspace
// layout and the launch. Everything here is plain host code around one kernel
// launch on the caller's stream; nothing synchronises with the device except
// pa_read_device_errors.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_params.h"

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t q) { return ceil_div(a, q) * q; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------- split plan
// Choose S (splits of each sequence's context) and P (tokens per split, a
// multiple of the warp tile: 16 tokens, 32 for fp8 caches, so that no tile
// crosses from one split's tokens into the next). The unit of parallel work is a (sequence,
// KV head, split) CTA, one resident per SM. The cost of a plan is the number of
// CTA waves times the tokens a CTA streams plus its fixed cost; candidates are
// one split, the largest split counts that fill exactly 1..4 waves, and 2..4
// splits (which can shorten the last wave when there are more (sequence, KV head)
// pairs than SMs).
struct Plan {
  int S;
  int P;
};

// A CTA's fixed cost (launch, first round trip, epilogue) expressed as the KV bytes
// it could have streamed meanwhile; the cost model charges it once per CTA and wave.
// Swept on GB300 (128 KiB .. 1 MiB): 256 KiB gave the best GQA grid and mixed batch,
// and the fewest wrong picks against ~60 forced-split timings (B = 1..64).
#ifndef PA_SPLIT_OVERHEAD_BYTES
#define PA_SPLIT_OVERHEAD_BYTES (256 << 10)
#endif
constexpr int64_t kSplitOverheadBytes = PA_SPLIT_OVERHEAD_BYTES;
#ifndef PA_PLAN_BALANCED
#define PA_PLAN_BALANCED 1
#endif

bool plan_for(int64_t S_req, int64_t max_len, int64_t p_max, bool floor_p, int64_t quantum,
              Plan* out) {
  int64_t P = round_up(ceil_div(max_len, std::max<int64_t>(S_req, 1)), quantum);
  if (floor_p) P = std::max<int64_t>(P, pa::kPartitionMin);
  P = std::min(P, p_max);
  int64_t S = ceil_div(max_len, P);
  if (S > pa::kMaxSplits) {
    P = round_up(ceil_div(max_len, pa::kMaxSplits), quantum);
    if (P > p_max) return false;  // context too long for this block size
    S = ceil_div(max_len, P);
  }
  *out = {(int)S, (int)P};
  return true;
}

bool make_plan(int sm_count, int64_t B, int64_t Hkv, int64_t D, int64_t kv_elem_bytes,
               int64_t max_len, int requested, int64_t quantum, int64_t total_tokens,
               Plan* out) {
  if (max_len <= 0) {
    *out = {1, (int)quantum};
    return true;
  }
  const int64_t units = B * Hkv;
  const int64_t sm = sm_count > 0 ? sm_count : 1;
  const int64_t p_max = round_up(max_len, quantum);
  if (requested > 0) return plan_for(requested, max_len, p_max, false, quantum, out);
  bool found = false;
  int64_t best_cost = 0;
  const int64_t cands[9] = {1, sm / units, 2 * sm / units, 3 * sm / units, 4 * sm / units,
                            ceil_div(sm, units), 2, 3, 4};
  // CTAs with tokens to stream: every split of every pair when the lengths are
  // unknown (all taken as max_len); given the batch's total context tokens, the
  // splits past each sequence's end are estimated away (a sequence's last split
  // counted as half full on average).
  auto live_ctas = [&](const Plan& pl) -> int64_t {
    const int64_t all = units * pl.S;
    if (total_tokens <= 0) return all;
    return std::min(all, Hkv * (ceil_div(total_tokens, pl.P) + ceil_div(B, 2)));
  };
  // A CTA streams its split as rounds of one tile per warp, so with a 16-bit cache
  // its time follows the tokens rounded up to whole rounds; a split of that rounded
  // size is as fast and needs fewer CTAs, which is also tried for every candidate.
  // An fp8 CTA is bound by its SM's instruction issue, so its time follows all its
  // tiles: no rounding there (rounded, the fp8 grid and hybrid steps lost 0.5-1%).
  const int64_t round_tokens =
      quantum * (PA_PLAN_BALANCED && kv_elem_bytes == 2 ? pa::warps_per_cta((int)D, false) : 1);
  auto consider = [&](const Plan& pl) {
    const int64_t waves = ceil_div(live_ctas(pl), sm);
    // the fixed cost in tokens of this cache: K + V bytes per token per KV head
    const int64_t overhead_tokens = kSplitOverheadBytes / (2 * D * kv_elem_bytes);
    const int64_t cost = waves * (round_up(pl.P, round_tokens) + overhead_tokens);
    if (!found || cost < best_cost || (cost == best_cost && pl.S < out->S)) {
      *out = pl;
      best_cost = cost;
      found = true;
    }
  };
  for (int64_t c : cands) {
    if (c < 1) continue;
    Plan pl{};
    if (!plan_for(c, max_len, p_max, true, quantum, &pl)) continue;
    consider(pl);
    const int64_t pr = std::min(round_up(pl.P, round_tokens), p_max);
    if (pr != pl.P) consider(Plan{(int)ceil_div(max_len, pr), (int)pr});
  }
  return found;
}

// ---------------------------------------------------------------- workspace
// [0, 256)            device error word (uint32) + padding
// [256, kHeaderBytes)  shared-tile counters, one int per (sequence, KV head)
// m, l                 B*Hkv*S*G fp32 each        (only when S > 1)
// acc        B*Hkv*S*G*D fp32           (only when S > 1)
struct WsLayout {
  size_t m, l, acc, total;
};

WsLayout ws_layout(int64_t B, int64_t Hkv, int64_t G, int64_t D, int64_t S) {
  WsLayout w{};
  size_t off = pa::kHeaderBytes;
  if (S > 1) {
    const size_t parts = (size_t)(B * Hkv * S * G);
    w.m = off;
    off += align256(parts * 4);
    w.l = off;
    off += align256(parts * 4);
    w.acc = off;
    off += align256(parts * (size_t)D * 4);
  }
  w.total = off;
  return w;
}

int current_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

// Size checks shared by the size query, the plan and the launch.
pa_status check_sizes(const pa_decode_args* a, int64_t* max_len) {
  if (a->B < 0) return PA_ERR_INVALID_ARG;
  if (a->Hq <= 0 || a->Hkv <= 0 || a->D <= 0) return PA_ERR_INVALID_ARG;
  if (a->Hq % a->Hkv != 0) return PA_ERR_INVALID_ARG;
  if (a->Hq / a->Hkv > PA_MAX_GQA_GROUP) return PA_ERR_INVALID_ARG;
  if (a->D != 128 && a->D != 256) return PA_ERR_UNSUPPORTED;
  if (a->block_size <= 0 || a->num_blocks <= 0 || a->max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  if (a->dtype != PA_F16 && a->dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (a->splits < 0 || a->window < 0 || a->q_len < 0) return PA_ERR_INVALID_ARG;
  {
    const int64_t rows = a->q_len > 0 ? a->q_len : 1;
    const int64_t cols = (int64_t)(a->Hq / a->Hkv) * rows;
    if (rows > 1 && a->window > 0) return PA_ERR_UNSUPPORTED;        // one or the other
    if (cols > (a->D == 128 ? 32 : 16)) return PA_ERR_UNSUPPORTED;    // (rows x group) per CTA
    if ((int64_t)a->Hq * rows > 65535) return PA_ERR_INVALID_ARG;     // merge grid limit
  }
  if (a->kv_dtype != PA_KV_AS_DTYPE && a->kv_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
  if (a->flags & ~PA_FLAG_DETERMINISTIC) return PA_ERR_INVALID_ARG;
  if (a->total_tokens < 0) return PA_ERR_INVALID_ARG;
  if (a->kv_dtype == PA_KV_FP8_E4M3 &&
      !(a->k_scale > 0.f && a->v_scale > 0.f && a->k_scale < INFINITY && a->v_scale < INFINITY))
    return PA_ERR_INVALID_ARG;
  if (a->B > 65535 || a->Hkv > 65535) return PA_ERR_INVALID_ARG;  // grid limits
  // kernels address cache rows with 32-bit row indices
  if ((int64_t)a->num_blocks * a->block_size * a->Hkv > (int64_t)UINT32_MAX) return PA_ERR_UNSUPPORTED;
  const int64_t cap = (int64_t)a->max_blocks_per_seq * a->block_size;
  int64_t ml = a->max_seq_len <= 0 ? cap : a->max_seq_len;
  if (ml > cap) return PA_ERR_OUT_OF_RANGE;
  if (ml > INT_MAX) return PA_ERR_OUT_OF_RANGE;
  if (a->total_tokens > (int64_t)a->B * ml) return PA_ERR_INVALID_ARG;  // contradicts max_seq_len
  *max_len = ml;
  return PA_OK;
}

// Bytes of one cache element.
int64_t kv_elem_bytes(const pa_decode_args* a) { return a->kv_dtype == PA_KV_FP8_E4M3 ? 1 : 2; }

// Tokens per warp tile of the kernel that serves these arguments.
int64_t tile_tokens(const pa_decode_args* a) {
  return pa::tile_tokens(a->D, a->kv_dtype == PA_KV_FP8_E4M3);
}

// The batch's total context tokens for the planner (0: unknown). A window bounds
// each sequence's tokens in a way the total does not tell, so it is not used then.
int64_t plan_tokens(const pa_decode_args* a) { return a->window > 0 ? 0 : a->total_tokens; }

// Tokens one sequence's splits must cover: a sliding window bounds them.
int64_t plan_len(const pa_decode_args* a, int64_t max_len) {
  return (a->window > 0 && a->window < max_len) ? a->window : max_len;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

const char* pa_version(void) { return "0.1.0"; }

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_OUT_OF_RANGE: return "value out of range";
  }
  return "unknown status";
}

pa_status pa_set_device(int device) {
  if (cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  return PA_OK;
}

// Division by the block size as a multiply-high and a shift (division by invariant
// integers using multiplication, Granlund and Montgomery, 1994): for d not a power
// of two, with l = ceil(log2 d), s = l - 1 and m = ceil(2^(32+s) / d) < 2^32,
// floor(n m / 2^(32+s)) = floor(n / d) for every 0 <= n < 2^31, since the error
// n (m d - 2^(32+s)) / (d 2^(32+s)) < 2^31 d / (d 2^(32+s)) <= 1/d.
static void set_block_division(int d, uint32_t* magic, int* shift) {
  int l = 0;
  while ((1ll << l) < d) ++l;  // ceil(log2 d)
  if ((1ll << l) == d) {       // a power of two: a shift
    *magic = 0;
    *shift = l;
    return;
  }
  const int s = l - 1;
  const unsigned long long num = 1ull << (32 + s);
  *magic = (uint32_t)((num + (unsigned long long)d - 1) / (unsigned long long)d);
  *shift = s;
}

pa_status pa_decode_plan(const pa_decode_args* a, int sm_count, int* splits,
                         int* partition_tokens) {
  if (!a || !splits || !partition_tokens) return PA_ERR_INVALID_ARG;
  int64_t max_len = 0;
  const pa_status st = check_sizes(a, &max_len);
  if (st != PA_OK) return st;
  if (sm_count <= 0) sm_count = current_sm_count();
  if (sm_count <= 0) return PA_ERR_CUDA;
  Plan plan{};
  if (!make_plan(sm_count, a->B, a->Hkv, a->D, kv_elem_bytes(a), plan_len(a, max_len), a->splits,
                 tile_tokens(a), plan_tokens(a), &plan))
    return PA_ERR_UNSUPPORTED;
  *splits = plan.S;
  *partition_tokens = plan.P;
  return PA_OK;
}

size_t pa_decode_ex_workspace_bytes(const pa_decode_args* a) {
  int S = 0, P = 0;
  if (pa_decode_plan(a, 0, &S, &P) != PA_OK) return 0;
  const int rows = a->q_len > 0 ? a->q_len : 1;
  return ws_layout(a->B, a->Hkv, (int64_t)(a->Hq / a->Hkv) * rows, a->D, S).total;
}

size_t pa_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int max_seq_len) {
  // The plan depends on the sizes and the longest context, not on how the context is
  // paged: any block size gives the same workspace, so one token per block stands in.
  if (max_seq_len <= 0) return 0;
  pa_decode_args a{};
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.block_size = 1;
  a.num_blocks = 1;
  a.max_blocks_per_seq = max_seq_len;
  a.max_seq_len = max_seq_len;
  a.dtype = PA_BF16;
  return pa_decode_ex_workspace_bytes(&a);
}

pa_status pa_workspace_init(void* workspace, size_t bytes, pa_stream_t stream) {
  if (!workspace) return PA_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  return PA_OK;
}

pa_status pa_read_device_errors(void* workspace, pa_stream_t stream, uint32_t* flags) {
  if (!workspace || !flags) return PA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(workspace, 0, sizeof(v), st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  *flags = v;
  return PA_OK;
}

// The decode call, or (kernels != nullptr) only the count of kernels it would launch:
// then no pointer is read and nothing is launched.
static pa_status decode_ex(const pa_decode_args* a, void* workspace, size_t workspace_bytes,
                           pa_stream_t stream, int* kernels) {
  if (!a) return PA_ERR_INVALID_ARG;
  int64_t max_len = 0;
  pa_status st = check_sizes(a, &max_len);
  if (st != PA_OK) return st;
  if (a->B == 0) {  // nothing to compute
    if (kernels) *kernels = 0;
    return PA_OK;
  }
  if (!kernels) {
    if (!a->q || !a->k_cache || !a->v_cache || !a->block_tables || !a->seq_lens || !a->out)
      return PA_ERR_INVALID_ARG;
    if (!aligned16(a->q) || !aligned16(a->k_cache) || !aligned16(a->v_cache) || !aligned16(a->out))
      return PA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PA_ERR_WORKSPACE;
  }

  const int sm = current_sm_count();
  if (sm <= 0) return PA_ERR_CUDA;
  Plan plan{};
  if (!make_plan(sm, a->B, a->Hkv, a->D, kv_elem_bytes(a), plan_len(a, max_len), a->splits,
                 tile_tokens(a), plan_tokens(a), &plan))
    return PA_ERR_UNSUPPORTED;
  const int G = a->Hq / a->Hkv;
  const int rows = a->q_len > 0 ? a->q_len : 1;
  const WsLayout w = ws_layout(a->B, a->Hkv, (int64_t)G * rows, a->D, plan.S);
  if (!kernels && workspace_bytes < w.total) return PA_ERR_WORKSPACE;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  pa::DecodeParams p{};
  p.q = a->q;
  p.k_cache = a->k_cache;
  p.v_cache = a->v_cache;
  p.block_tables = a->block_tables;
  p.seq_lens = a->seq_lens;
  p.out = a->out;
  p.err = reinterpret_cast<uint32_t*>(ws);
  p.ws_m = plan.S > 1 ? reinterpret_cast<float*>(ws + w.m) : nullptr;
  p.ws_l = plan.S > 1 ? reinterpret_cast<float*>(ws + w.l) : nullptr;
  p.ws_acc = plan.S > 1 ? reinterpret_cast<float*>(ws + w.acc) : nullptr;
  p.B = a->B;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.G = G;
  p.block_size = a->block_size;
  set_block_division(a->block_size, &p.bs_magic, &p.bs_shift);
  p.num_blocks = a->num_blocks;
  p.max_blocks = a->max_blocks_per_seq;
  p.max_seq_len = (int)max_len;
  p.S = plan.S;
  p.P = plan.P;
  // static share per split; the rest of each context is claimed tile by tile
  p.Ps = plan.P;
  const long long split_bytes = (long long)plan.P * 2 * a->D * (a->kv_dtype == PA_KV_FP8_E4M3 ? 1 : 2);
  if (plan.S > 1 && !(a->flags & PA_FLAG_DETERMINISTIC) && pa::kStealDiv > 0 &&
      split_bytes >= pa::kStealMinBytes && (int64_t)a->B * a->Hkv <= pa::kStealUnits) {
    const int tw = (int)tile_tokens(a);  // static shares stay whole tiles
    const int shared = (plan.P / pa::kStealDiv) / tw * tw;
    p.Ps = plan.P - shared;
  }
  p.steal = reinterpret_cast<int*>(ws + 256);
  p.window = a->window;
  p.q_len = rows;
  p.kv_fp8 = a->kv_dtype == PA_KV_FP8_E4M3;
  p.v_scale = p.kv_fp8 ? a->v_scale : 1.f;
  // scores live in the exp2 domain; an fp8 K's scale multiplies every score
  p.scale_log2 = (float)((double)a->scale * 1.4426950408889634 * (p.kv_fp8 ? (double)a->k_scale : 1.0));

  cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e;
  const bool bf16 = a->dtype == PA_BF16;
  if (p.kv_fp8) {
    if (a->D == 128)
      e = bf16 ? pa::launch_decode_fp8_bf16_d128(p, cs, kernels) : pa::launch_decode_fp8_f16_d128(p, cs, kernels);
    else
      e = bf16 ? pa::launch_decode_fp8_bf16_d256(p, cs, kernels) : pa::launch_decode_fp8_f16_d256(p, cs, kernels);
  } else if (a->D == 128) {
    e = bf16 ? pa::launch_decode_bf16_d128(p, cs, kernels) : pa::launch_decode_f16_d128(p, cs, kernels);
  } else {
    e = bf16 ? pa::launch_decode_bf16_d256(p, cs, kernels) : pa::launch_decode_f16_d256(p, cs, kernels);
  }
  if (e != cudaSuccess && kernels) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    // A grid of this call may already be queued (the decode grid, when a later launch
    // failed) and would leave its tile counters claimed: clear the header behind it
    // on the same stream, so that the workspace still serves the next call.
    if (cudaMemsetAsync(workspace, 0, pa::kHeaderBytes, cs) != cudaSuccess) cudaGetLastError();
    return PA_ERR_CUDA;
  }
  return PA_OK;
}

pa_status pa_decode_ex(const pa_decode_args* a, void* workspace, size_t workspace_bytes,
                       pa_stream_t stream) {
  return decode_ex(a, workspace, workspace_bytes, stream, nullptr);
}

pa_status pa_decode_kernel_count(const pa_decode_args* a, int* kernels) {
  if (!kernels) return PA_ERR_INVALID_ARG;
  return decode_ex(a, nullptr, 0, nullptr, kernels);
}

pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* seq_lens, void* out, int B,
                    int Hq, int Hkv, int D, int block_size, int num_blocks,
                    int max_blocks_per_seq, int max_seq_len, float scale, pa_dtype dtype,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream) {
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
  return pa_decode_ex(&a, workspace, workspace_bytes, stream);
}

}  // extern "C"

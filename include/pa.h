/*
 * pa.h -- C ABI of libpa.so: single-query paged-attention decode on GB300 (sm_103a).
 *
 * The operation. "vLLM's custom ROCm paged-attention kernel wins all sixty cells"
 * (gqa-gate-costs-nothing), section 1, states the problem: pure decode, one query
 * token per sequence and head, attending over a fully cached context. The context
 * lives in a block-paged K/V cache addressed through a block table. For sequence b
 * of length L = seq_lens[b], query head h and its KV head g(h) = h / G (G = Hq/Hkv):
 *
 *   s_t      = scale * dot(q[b,h,:], K[b,t,g(h),:])            t < L
 *   out[b,h] = sum_t softmax(s)_t * V[b,t,g(h),:]
 *
 * where token t of sequence b is row (t % block_size) of physical block
 * block_tables[b][t / block_size]. Slots at or past L (the unwritten tail of the
 * last block, section 5 of the same page) are never read, so NaN there cannot
 * reach the output. The context is split across CTAs and merged afterwards (the
 * split-KV fix in "Hybrid-SSM decode rate on dual Radeon cards under vLLM"),
 * with fp32 accumulation throughout and one rounding to the output type.
 *
 * Conventions for every call below.
 *  - Pointers named q, k_cache, v_cache, block_tables, seq_lens, out, workspace
 *    are DEVICE pointers, owned by the caller; the library never allocates, frees
 *    or retains them, and keeps no state between calls.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) on the device current to the calling thread inside this library
 *    (see pa_set_device). Host-side argument errors are returned synchronously
 *    and nothing is launched.
 *  - Kernels are launched with programmatic stream serialization. Each one waits
 *    for the kernel before it in the stream to complete (griddepcontrol.wait)
 *    before reading any input, so inputs written by that kernel are safe. Each
 *    one also lets the next kernel in the stream start early: a kernel that the
 *    caller launches after a decode call with the programmatic-serialization
 *    attribute must wait in the same way (cudaGridDependencySynchronize) before
 *    it reads `out`; a kernel launched without the attribute needs nothing.
 *  - Layouts are dense, row-major, with no padding:
 *        q, out        [B, Hq, D]                       (dtype)
 *        k_cache,
 *        v_cache       [num_blocks, block_size, Hkv, D] (dtype)
 *        block_tables  [B, max_blocks_per_seq]          int32
 *        seq_lens      [B]                              int32
 *    q, k_cache, v_cache and out must be 16-byte aligned.
 *  - Device-side problems (a block table entry outside [0, num_blocks) for a live
 *    token, a seq_len that is negative or above max_seq_len or above
 *    max_blocks_per_seq*block_size) never fault:
 *    the kernel clamps, keeps going, and ORs a PA_DEVERR_* bit into the workspace
 *    header; read it with pa_read_device_errors. The output of such a call is
 *    finite but not meaningful.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, Hq % Hkv != 0, G > 16 */
  PA_ERR_UNSUPPORTED = 2,   /* head_dim not 128/256, or an option this build does not implement */
  PA_ERR_WORKSPACE = 3,     /* workspace too small or misaligned */
  PA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed (the CUDA error is cleared) */
  PA_ERR_OUT_OF_RANGE = 5   /* max_seq_len above max_blocks_per_seq * block_size, or a device error */
} pa_status;

typedef enum pa_dtype { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

/* Element type of the K/V caches in pa_decode_args.kv_dtype. */
typedef enum pa_kv_dtype {
  PA_KV_AS_DTYPE = 0, /* the caches have the q/out dtype */
  PA_KV_FP8_E4M3 = 1  /* FP8 E4M3 ("fn": bias 7, no infinities, max 448), one byte per
                         element; cache value = stored value * k_scale (K) or v_scale (V) */
} pa_kv_dtype;

/* Bits of the device error word (workspace header). */
#define PA_DEVERR_BLOCK_INDEX 1u /* a live token's block table entry was outside [0, num_blocks) */
#define PA_DEVERR_SEQ_LEN 2u     /* a seq_len < 0, > max_seq_len or > max_blocks_per_seq*block_size */

typedef void* pa_stream_t; /* cudaStream_t */

/* Largest query-head group (Hq / Hkv) a call accepts. */
#define PA_MAX_GQA_GROUP 16

/*
 * Full argument set for pa_decode_ex. Fields beyond those of pa_decode:
 *   splits  0 = choose the split count automatically (fill every SM even at batch 1);
 *           > 0 = use at most this many splits of the context (tests, tuning).
 *   window  0 = attend to the whole context; > 0 = sliding-window decode: each
 *           query attends to the last `window` tokens of its context, t in
 *           [max(0, L - window), L) (the sliding layers of "vLLM's custom ROCm
 *           paged-attention kernel wins all sixty cells", section 4, scan 1024).
 *           Table entries before the window are not read.
 *   kv_dtype  PA_KV_AS_DTYPE (default) or PA_KV_FP8_E4M3: the caches hold one byte
 *           per element, [num_blocks, block_size, Hkv, D] as before; q and out keep
 *           `dtype`. fp8 K/V are widened exactly to fp16 for the tensor-core
 *           products (the queries are rounded to fp16, so bf16 query elements must
 *           lie within fp16's range, |x| <= 65504; P is kept in fp16) with fp32
 *           accumulation. The pages list an fp8 cache as untested ("vLLM's custom
 *           ROCm paged-attention kernel wins all sixty cells", section 6).
 *   k_scale, v_scale  per-tensor dequantisation scales (finite, > 0) for an fp8
 *           cache; ignored otherwise.
 *   q_len   query rows per sequence (0 or 1 = single-query decode). With R > 1 rows,
 *           q and out are [B, R, Hq, D]: row i is the query of token L - R + i (the
 *           new tokens of a speculative-decode step or a chunked-prefill tail) and
 *           attends causally to the tokens t < L - R + i + 1; a row that sees no
 *           token gets zeros. Every K/V tile is read once for all rows and heads of
 *           its KV head. Limits: G * R <= 32 at head_dim 128, <= 16 at 256; not
 *           combined with a window (PA_ERR_UNSUPPORTED).
 *   flags   0 or PA_FLAG_DETERMINISTIC. By default, when a long context is split
 *           across CTAs, the splits share out its last eighth tile by tile as
 *           they finish their own shares, so the order of the fp32 sums depends
 *           on timing and repeated calls may differ in the last bit (each within
 *           the usual error). PA_FLAG_DETERMINISTIC keeps fixed splits: repeated
 *           calls give bitwise identical outputs. Other bits: PA_ERR_INVALID_ARG.
 *   total_tokens  0, or the sum of seq_lens over the batch, known on the host like
 *           max_seq_len. It lets the planner estimate how many context splits hold
 *           tokens in a batch of mixed lengths; only the split plan depends on it
 *           (a wrong value costs speed, not correctness). Negative, or above
 *           B * max_seq_len: PA_ERR_INVALID_ARG. Ignored with a window.
 * All other fields mean what the pa_decode parameters of the same name mean.
 */
typedef struct pa_decode_args {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  void* out;
  int32_t B, Hq, Hkv, D;
  int32_t block_size, num_blocks, max_blocks_per_seq, max_seq_len;
  float scale;
  int32_t dtype; /* pa_dtype */
  int32_t splits;
  int32_t window;
  int32_t kv_dtype; /* pa_kv_dtype */
  float k_scale, v_scale;
  int32_t q_len;
  uint32_t flags;
  int64_t total_tokens;
} pa_decode_args;

#define PA_FLAG_DETERMINISTIC 1u

/*
 * Workspace bytes pa_decode needs for these sizes on the current device (the
 * problem's sizes and the host-side bound on seq_lens; the split plan does not
 * depend on the block size, so the query does not take one). The
 * workspace starts with a header of PA_WORKSPACE_HEADER_BYTES that must be zero
 * before the first call (pa_workspace_init or any memset): the device error word
 * (first 4 bytes) and one counter per (sequence, KV head) through which the
 * splits of a sequence share out the tail of its context; every call leaves the
 * counters zero again. After the header come the fp32 split partials (m, l, acc),
 * which every call writes before it reads them. One workspace serves calls of
 * any shape that fit its size; calls that overlap on the GPU must not share one.
 * Returns 0 for invalid sizes (max_seq_len must be > 0 here).
 */
#define PA_WORKSPACE_HEADER_BYTES 8448u
size_t pa_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int max_seq_len);

/* Same, for pa_decode_ex's argument set (pointer fields are ignored). */
size_t pa_decode_ex_workspace_bytes(const pa_decode_args* args);

/*
 * Single-query paged-attention decode: the call of the problem statement in "vLLM's
 * custom ROCm paged-attention kernel wins all sixty cells" (gqa-gate-costs-nothing),
 * section 1 (one query token per sequence and head over a fully cached, block-paged
 * context), with the split-KV partition and reduce of "Hybrid-SSM decode rate on dual
 * Radeon cards under vLLM" (its split-KV paragraph) chosen inside the call.
 *   q             [B, Hq, D] queries (dtype)
 *   k_cache,
 *   v_cache       [num_blocks, block_size, Hkv, D] paged keys / values (dtype)
 *   block_tables  [B, max_blocks_per_seq] int32 physical block of each logical block;
 *                 entries past ceil(seq_lens[b] / block_size) are never read
 *   seq_lens      [B] int32 context length per sequence (0 gives a zero output row)
 *   out           [B, Hq, D] output (dtype), fully written
 *   B             batch (0 is a no-op), Hq and Hkv query and KV heads (Hq % Hkv == 0,
 *                 Hq / Hkv <= PA_MAX_GQA_GROUP), D head_dim (128 or 256)
 *   block_size    tokens per block (any positive size, e.g. 16 or 784)
 *   num_blocks    blocks in each cache tensor
 *   max_seq_len   a host-side upper bound on seq_lens (used to choose the split
 *                 count without reading device memory); <= 0 means
 *                 max_blocks_per_seq * block_size
 *   scale         softmax scale applied to q.k (e.g. 1/sqrt(D))
 *   dtype         PA_F16 or PA_BF16 for q, caches and out
 *   workspace     device scratch of >= pa_decode_workspace_bytes(...) bytes,
 *                 256-byte aligned, its header zero before first use
 * Errors: PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE,
 * PA_ERR_OUT_OF_RANGE (max_seq_len above capacity), PA_ERR_CUDA. On PA_ERR_CUDA a
 * kernel of the call may already be queued; the call then also queues, behind it on
 * `stream`, a clearing of the workspace header (tile counters and device error word),
 * so that the workspace stays usable if the context does.
 */
pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* seq_lens, void* out,
                    int B, int Hq, int Hkv, int D, int block_size, int num_blocks,
                    int max_blocks_per_seq, int max_seq_len, float scale, pa_dtype dtype,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream);

/* pa_decode with the extra options of pa_decode_args. Same errors. */
pa_status pa_decode_ex(const pa_decode_args* args, void* workspace, size_t workspace_bytes,
                       pa_stream_t stream);

/*
 * The launch plan pa_decode_ex would use on a GPU with `sm_count` SMs: the number
 * of context splits and the tokens per split, a whole number of warp tiles (32
 * tokens at head_dim 128 and for fp8 caches, 16 at head_dim 256). It depends on the
 * sizes, max_seq_len, window, kv_dtype, splits and total_tokens of `args`. Pure
 * host arithmetic; needs no GPU. sm_count <= 0 means the current device's SM count.
 */
pa_status pa_decode_plan(const pa_decode_args* args, int sm_count, int* splits,
                         int* partition_tokens);

/*
 * How many kernels pa_decode_ex would launch for `args` on the current device (the
 * plan, and whether the splits merge inside their thread-block clusters, depend on
 * the device): 0 for B == 0, 1 for a context in one split or splits that merge in
 * their cluster, 2 for a decode grid followed by a merge grid. Pointer fields are
 * not read; nothing is launched. The same argument errors as pa_decode_ex.
 */
pa_status pa_decode_kernel_count(const pa_decode_args* args, int* kernels);

/* Zero-fill a workspace on `stream` (asynchronous). */
pa_status pa_workspace_init(void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * Wait for `stream`, then copy the device error word (PA_DEVERR_* bits) of
 * `workspace` to *flags and clear it. Synchronous.
 */
pa_status pa_read_device_errors(void* workspace, pa_stream_t stream, uint32_t* flags);

/* Make `device` current for this library's calls on the calling thread. */
pa_status pa_set_device(int device);

/*
 * pa_decode without a workspace, for callers that cannot allocate device memory
 * or pass scratch to the library: for example a plugin inside another runtime
 * that owns all device allocations, code that must not call cudaMalloc because
 * it may synchronise the device, or a binding with no device allocator. The pages
 * describe no such call; it exists only for those callers.
 *
 * Arguments, layouts, validation and results are those of pa_decode. The split
 * partials live in one array of PA_NOALLOC_SCRATCH_BYTES that is part of this
 * library's device image: every GPU that loads it keeps that memory until the
 * process exits, and the call itself allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *  - Limit: a call whose partials need more than PA_NOALLOC_SCRATCH_BYTES (as
 *    pa_decode_workspace_bytes reports) returns PA_ERR_WORKSPACE and launches
 *    nothing; use pa_decode with your own workspace for it.
 *  - The first call on a device looks up the array's device address (once, kept
 *    for the life of the process) and clears the array's header with an
 *    asynchronous memset on `stream`, ordered before that call's kernels; make that
 *    first call before any stream capture on that device. The address belongs to
 *    the device's current context: after cudaDeviceReset on a device, this entry
 *    point must not be called on it again in the same process.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents. Nothing in it needs to start at zero except its header (the tile
 *    counters, which every successful call leaves at zero, and the error word).
 *    Calls that may overlap on the GPU (different streams, concurrent threads)
 *    race on it: serialise them. A call that returns PA_ERR_CUDA queues a clearing
 *    of the header on `stream`, as pa_decode does for its workspace.
 *  - Device-side range errors (PA_DEVERR_*) are recorded in the array's header
 *    and are not readable through this API.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)
pa_status pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* seq_lens, void* out,
                            int B, int Hq, int Hkv, int D, int block_size, int num_blocks,
                            int max_blocks_per_seq, int max_seq_len, float scale,
                            pa_dtype dtype, pa_stream_t stream);

/* Static text for a status code. */
const char* pa_status_string(pa_status status);

/* Library version, e.g. "0.1.0". */
const char* pa_version(void);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* PA_H_ */

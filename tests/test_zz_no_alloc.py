"""pa_decode_noalloc against pa_decode and the float64 oracle (GB300 only).

pa_decode_noalloc serves callers that cannot give the library device scratch
memory: a plugin inside a runtime that owns all device allocations, code that
must not call cudaMalloc (it can synchronise the device), a binding with no
device allocator. Its split partials and tile counters live in a fixed device
array of the library instead of a caller workspace.

Each case below needs several context splits, so the array is really used. Every
case is called twice in a row through the C ABI (the second call finds the first
call's partials and counters in the array); both outputs are held to the oracle
bar and to pa_decode's output. The first call of the file runs on a non-blocking
stream, where the array's first-use header clearing must be ordered before the
kernels on that stream. The file is collected last so that a failure here leaves
every other test run.
"""
import numpy as np
import pytest
import torch

import pa_inputs as pi
from harness import REL_LINF_TOL, assert_parity, oracle_case, oracle_rows
from oracle import rel_linf_error

pytestmark = pytest.mark.gpu


def _call_noalloc(pa, c, out, stream):
    lib = pa.load()
    a = pa.make_args(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, out, c.scale,
                     c.max_seq_len)
    pa._ensure_device(lib, c.q.device.index)
    return lib.pa_decode_noalloc(a.q, a.k_cache, a.v_cache, a.block_tables, a.seq_lens, a.out,
                                 a.B, a.Hq, a.Hkv, a.D, a.block_size, a.num_blocks,
                                 a.max_blocks_per_seq, a.max_seq_len, a.scale, a.dtype,
                                 stream.cuda_stream)


def _oracle(case, full):
    """Float64 oracle output [B, Hq, D]: every (sequence, KV head) when `full`, else
    KV heads 0 and Hkv - 1 of every sequence (NaN elsewhere, not compared)."""
    if full:
        return oracle_case(case)
    G = case.Hq // case.Hkv
    ref = np.full((case.B, case.Hq, case.D), np.nan)
    pairs = [(b, h) for b in range(case.B) for h in {0, case.Hkv - 1}]
    for (b, h), r in oracle_rows(case, pairs).items():
        ref[b, h * G:(h + 1) * G] = r
    return ref


def _check(y, ref, what):
    keep = ~np.isnan(ref[:, :, 0])
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    return assert_parity(y[keep], ref[keep], what=what)


def test_noalloc_matches_oracle_and_workspace_entry_point(cuda_lib):
    pa = cuda_lib
    cases = [
        # (case, compare every output against the oracle)
        (pi.make_case(1, 24, 4, 256, 784, [5000], seed=31, poison="kv_nan"), True),
        (pi.make_case(3, 32, 8, 128, 16, [4097, 1000, 2222], seed=32, poison="v_nan"), True),
        # long enough that the splits share the tail through the array's tile counters
        (pi.make_case(1, 8, 8, 128, 16, [32768], seed=34, poison="kv_nan", device="cuda"), False),
        (pi.make_case(1, 8, 8, 128, 16, [32000], seed=35, device="cuda"), False),
    ]
    side = torch.cuda.Stream()  # torch creates its side streams non-blocking
    for i, (case, full) in enumerate(cases):
        c = case.to("cuda")
        S, _ = pa.plan(c.B, c.Hq, c.Hkv, c.D, c.block_size, c.max_seq_len)
        assert S > 1, "the case must use split partials"
        ref = _oracle(case, full)
        want = pa.decode_plain(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, c.scale,
                               max_seq_len=c.max_seq_len)
        torch.cuda.synchronize()
        w = want.double().cpu().numpy()
        # the first case runs on a separate (non-blocking) stream, the others on the
        # current stream; two calls in a row each
        stream = side if i == 0 else torch.cuda.current_stream()
        for rep in range(2):
            out = torch.full_like(c.q, float("nan"))
            torch.cuda.synchronize()
            assert _call_noalloc(pa, c, out, stream) == pa.PA_OK
            stream.synchronize()
            y = out.double().cpu().numpy()
            _check(y, ref, f"noalloc case {i} call {rep + 1}")
            assert rel_linf_error(y, w) <= REL_LINF_TOL, f"case {i} call {rep + 1} vs pa_decode"


def test_noalloc_validates_like_pa_decode(cuda_lib):
    pa = cuda_lib
    lib = pa.load()
    c = pi.make_case(1, 8, 8, 128, 16, [100], seed=33).to("cuda")
    out = torch.empty_like(c.q)
    a = pa.make_args(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, out, c.scale, 100)
    st = torch.cuda.current_stream().cuda_stream
    common = (a.block_size, a.num_blocks, a.max_blocks_per_seq, a.max_seq_len, a.scale, a.dtype, st)
    # head_dim 64 is unsupported, Hq % Hkv != 0 is invalid, a null q is invalid
    assert lib.pa_decode_noalloc(a.q, a.k_cache, a.v_cache, a.block_tables, a.seq_lens, a.out,
                                 1, 8, 8, 64, *common) == pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode_noalloc(a.q, a.k_cache, a.v_cache, a.block_tables, a.seq_lens, a.out,
                                 1, 12, 8, 128, *common) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_noalloc(None, a.k_cache, a.v_cache, a.block_tables, a.seq_lens, a.out,
                                 1, 8, 8, 128, *common) == pa.PA_ERR_INVALID_ARG
    # A call whose partials exceed the fixed array is refused before any launch. The
    # sizes are checked on the host first, so that the call is only made with sizes
    # the library is known to refuse (its pointers belong to the small case above).
    shapes = [(B, 16 * hkv, hkv, 256, L) for B in (64, 128, 256) for hkv in (8, 16)
              for L in (1 << 16, 1 << 18, 1 << 20)]
    big = next((s for s in shapes if lib.pa_decode_workspace_bytes(*s) > pa.PA_NOALLOC_SCRATCH_BYTES),
               None)
    assert big is not None, "no shape needs more scratch than the fixed array"
    B, Hq, Hkv, D, L = big
    assert lib.pa_decode_noalloc(a.q, a.k_cache, a.v_cache, a.block_tables, a.seq_lens, a.out,
                                 B, Hq, Hkv, D, 16, 1, L // 16, L, a.scale, a.dtype,
                                 st) == pa.PA_ERR_WORKSPACE

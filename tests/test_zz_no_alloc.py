"""pa_decode_noalloc against pa_decode (GB300 only).

pa_decode_noalloc serves callers that cannot give the library device scratch
memory (a plugin inside a runtime that owns all device allocations, code that
must not call cudaMalloc, a binding with no device allocator): its split
partials live in a fixed device array of the library instead of a caller
workspace. This test calls it through the C ABI twice in a row, on cases that
need several context splits (so the array is really used, and the second call
finds the first call's partials in it), and compares each output with the
workspace entry point within the parity tolerance of the other GPU tests.
It is collected last so that a failure here leaves every other test run.
"""
import numpy as np
import pytest
import torch

import pa_inputs as pi
from harness import REL_LINF_TOL
from oracle import rel_linf_error

pytestmark = pytest.mark.gpu


def _call_noalloc(pa, c, out):
    lib = pa.load()
    a = pa.make_args(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, out, c.scale,
                     c.max_seq_len)
    pa._ensure_device(lib, c.q.device.index)
    rc = lib.pa_decode_noalloc(a.q, a.k_cache, a.v_cache, a.block_tables, a.seq_lens, a.out,
                               a.B, a.Hq, a.Hkv, a.D, a.block_size, a.num_blocks,
                               a.max_blocks_per_seq, a.max_seq_len, a.scale, a.dtype,
                               torch.cuda.current_stream().cuda_stream)
    return rc


def test_noalloc_matches_workspace_entry_point(cuda_lib):
    pa = cuda_lib
    cases = [
        pi.make_case(1, 24, 4, 256, 784, [5000], seed=31, poison="kv_nan").to("cuda"),
        pi.make_case(3, 32, 8, 128, 16, [4097, 1000, 2222], seed=32, poison="v_nan").to("cuda"),
        # long enough that the splits share the tail through the array's tile counters
        pi.make_case(1, 8, 8, 128, 16, [32768], seed=34, poison="kv_nan", device="cuda"),
        pi.make_case(1, 8, 8, 128, 16, [32000], seed=35, device="cuda"),
    ]
    for c in cases:
        S, _ = pa.plan(c.B, c.Hq, c.Hkv, c.D, c.block_size, c.max_seq_len)
        assert S > 1, "the case must use split partials"
    for c in cases:  # two calls in a row, each checked against pa_decode's output
        ref = pa.decode_plain(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, c.scale,
                              max_seq_len=c.max_seq_len)
        out = torch.full_like(c.q, float("nan"))
        assert _call_noalloc(pa, c, out) == pa.PA_OK
        torch.cuda.synchronize()
        y = out.double().cpu().numpy()
        r = ref.double().cpu().numpy()
        assert np.all(np.isfinite(y))
        assert rel_linf_error(y, r) <= REL_LINF_TOL


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

"""The C ABI on a machine without a GPU: the library loads, exports every symbol
include/pa.h declares, validates arguments on the host, and plans launches."""
import ctypes
import os
import re

import pytest

import paged_kv_attention_pa_gb300 as pa
from paged_kv_attention_pa_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return pa.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(pa_[a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 10, names
    for n in names:
        assert hasattr(lib, n), f"libpa.so does not export {n}"
    assert set(names) == set(pa.SIGNATURES), "binding signatures and header disagree"


def test_status_strings_and_version(lib):
    for code in range(6):
        assert pa.status_string(code)
    assert pa.status_string(99) == "unknown status"
    assert pa.version() == pa.__version__


def _args(**kw):
    a = pa.DecodeArgs()
    base = dict(q=16, k_cache=32, v_cache=48, block_tables=64, seq_lens=80, out=96,
                B=1, Hq=8, Hkv=8, D=128, block_size=16, num_blocks=64,
                max_blocks_per_seq=32, max_seq_len=512, scale=0.088, dtype=pa.PA_BF16, splits=0)
    base.update(kw)
    for k, v in base.items():
        setattr(a, k, v)
    return a


def _call(lib, a, ws=256, nbytes=1 << 20):
    return lib.pa_decode_ex(ctypes.byref(a), ws, nbytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=12, Hkv=8), pa.PA_ERR_INVALID_ARG),            # Hq % Hkv != 0
    (dict(Hq=34, Hkv=2), pa.PA_ERR_INVALID_ARG),            # G = 17 > 16
    (dict(D=64), pa.PA_ERR_UNSUPPORTED),
    (dict(D=0), pa.PA_ERR_INVALID_ARG),
    (dict(block_size=0), pa.PA_ERR_INVALID_ARG),
    (dict(num_blocks=0), pa.PA_ERR_INVALID_ARG),
    (dict(B=-1), pa.PA_ERR_INVALID_ARG),
    (dict(dtype=7), pa.PA_ERR_INVALID_ARG),
    (dict(splits=-2), pa.PA_ERR_INVALID_ARG),
    (dict(max_seq_len=513), pa.PA_ERR_OUT_OF_RANGE),        # above 32 blocks * 16
    (dict(q=0), pa.PA_ERR_INVALID_ARG),
    (dict(out=0), pa.PA_ERR_INVALID_ARG),
    (dict(k_cache=40), pa.PA_ERR_INVALID_ARG),              # not 16-byte aligned
    (dict(num_blocks=1 << 24, block_size=784, Hkv=8, Hq=8), pa.PA_ERR_UNSUPPORTED),  # rows > 2^32
    (dict(kv_dtype=7), pa.PA_ERR_INVALID_ARG),
    (dict(kv_dtype=pa.PA_KV_FP8_E4M3, k_scale=0.0, v_scale=1.0), pa.PA_ERR_INVALID_ARG),
    (dict(kv_dtype=pa.PA_KV_FP8_E4M3, k_scale=1.0, v_scale=float("inf")), pa.PA_ERR_INVALID_ARG),
    (dict(window=-1), pa.PA_ERR_INVALID_ARG),
    (dict(q_len=-1), pa.PA_ERR_INVALID_ARG),
    (dict(q_len=2, window=64), pa.PA_ERR_UNSUPPORTED),      # rows and a window: not both
    (dict(q_len=5, Hq=56, Hkv=8), pa.PA_ERR_UNSUPPORTED),   # 7 x 5 = 35 columns > 32
    (dict(q_len=3, Hq=48, Hkv=8, D=256), pa.PA_ERR_UNSUPPORTED),  # 18 columns > 16
    (dict(flags=2), pa.PA_ERR_INVALID_ARG),                 # unknown flag bit
    (dict(total_tokens=-1), pa.PA_ERR_INVALID_ARG),
    (dict(total_tokens=513), pa.PA_ERR_INVALID_ARG),         # above B * max_seq_len
])
def test_host_validation(lib, kw, code):
    assert _call(lib, _args(**kw)) == code


def test_workspace_checks_precede_cuda(lib):
    assert _call(lib, _args(), ws=0) == pa.PA_ERR_WORKSPACE
    assert _call(lib, _args(), ws=272) == pa.PA_ERR_WORKSPACE   # not 256-byte aligned


def test_workspace_header(lib):
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    m = re.search(r"#define PA_WORKSPACE_HEADER_BYTES (\d+)u", src)
    assert m and int(m.group(1)) == pa.PA_WORKSPACE_HEADER_BYTES
    assert pa.PA_WORKSPACE_HEADER_BYTES % 256 == 0
    # the header (error word + one tile counter per (sequence, KV head)) precedes the
    # split partials, whatever the call's shape
    import torch
    if torch.cuda.is_available():  # sizes follow the current device's SM count
        for B, Hkv, L in [(1, 8, 512), (1, 4, 32768), (64, 8, 32768)]:
            need = lib.pa_decode_workspace_bytes(B, 2 * Hkv, Hkv, 128, L)
            assert need >= pa.PA_WORKSPACE_HEADER_BYTES
    a = _args(flags=pa.PA_FLAG_DETERMINISTIC)
    assert lib.pa_decode_ex_workspace_bytes(ctypes.byref(a)) == \
        lib.pa_decode_ex_workspace_bytes(ctypes.byref(_args()))
    # a workspace of exactly the header is too small for a call that splits
    assert _call(lib, _args(max_seq_len=512), nbytes=pa.PA_WORKSPACE_HEADER_BYTES) in (
        pa.PA_ERR_WORKSPACE, pa.PA_ERR_CUDA)


def test_empty_batch_is_a_noop(lib):
    assert _call(lib, _args(B=0, q=0, out=0)) == pa.PA_OK


def test_valid_call_without_gpu_reports_cuda(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call(lib, _args()) == pa.PA_ERR_CUDA


def test_plain_entry_point_validates(lib):
    rc = lib.pa_decode(16, 32, 48, 64, 80, 96, 1, 12, 8, 128, 16, 64, 32, 512, 0.1,
                       pa.PA_BF16, 256, 1 << 20, None)
    assert rc == pa.PA_ERR_INVALID_ARG


# ------------------------------------------------------------------ planner
SM = 152


@pytest.mark.parametrize("B,Hkv,bs,L", [
    (1, 8, 16, 512), (1, 4, 784, 4096), (1, 4, 784, 32768), (1, 8, 16, 1024),
    (8, 16, 16, 32768), (64, 8, 16, 32768), (1, 1, 1, 300000), (5, 8, 16, 16385),
    (1, 4, 784, 500), (2, 3, 7, 1000),
])
def test_plan_properties(lib, B, Hkv, bs, L):
    S, P = pa.plan(B, Hkv * 2, Hkv, 128, bs, L, sm_count=SM)
    assert P % 16 == 0 and P > 0
    assert S * P >= L, "the splits cover the longest context"
    assert (S - 1) * P < L, "no split of the longest context is empty"
    assert S <= 1024
    # many waves only with few splits (more (sequence, KV head) pairs than SMs)
    waves = -(-B * Hkv * S // SM)
    assert waves <= 4 or S <= 4


def test_plan_fills_sms_at_batch_one():
    # one wave, every warp of a CTA streaming the same number of 16-token tiles
    # (4 warps: splits of whole 64-token rounds)
    S, P = pa.plan(1, 24, 4, 256, 784, 32768, sm_count=SM)
    assert (S, P) == (37, 896) and 4 * S <= SM
    S, P = pa.plan(1, 24, 4, 256, 784, 4096, sm_count=SM)
    assert (S, P) == (32, 128)


def test_plan_rounds_splits_to_whole_warp_rounds():
    # A split of 7 tiles keeps three warps busy for two tiles and one for one; 8 tiles
    # take as long on fewer CTAs (GB300, us per call: 8/8 heads at batch 1, 4K: 6.60
    # for 16 splits of 256 tokens against 6.87 for 19 of 224; 8K: 9.11 against 9.87;
    # the hybrid layer at 8K: 10.01 for 32 splits of 256 against 10.57 for 38 of 224)
    assert pa.plan(1, 8, 8, 128, 16, 4096, sm_count=SM) == (16, 256)
    assert pa.plan(1, 8, 8, 128, 16, 8192, sm_count=SM) == (16, 512)
    assert pa.plan(1, 24, 4, 256, 784, 8192, sm_count=SM) == (32, 256)
    for B, Hkv, D, L in [(1, 8, 128, 4096), (1, 4, 256, 12288), (8, 8, 128, 16384)]:
        S, P = pa.plan(B, 2 * Hkv, Hkv, D, 16, L, sm_count=SM)
        assert P % (4 * (32 if D == 128 else 16)) == 0 and S * P >= L


def test_forced_splits():
    for want in (1, 2, 3, 7):
        S, P = pa.plan(1, 16, 8, 128, 16, 1025, splits=want, sm_count=SM)
        assert S == want and S * P >= 1025
    # the finest split is one warp tile: 32 tokens at head_dim 128 and for fp8
    # caches, 16 at head_dim 256
    S, P = pa.plan(1, 16, 8, 128, 16, 1025, splits=10000, sm_count=SM)
    assert P == 32 and S == 33
    S, P = pa.plan(1, 16, 8, 256, 16, 1025, splits=10000, sm_count=SM)
    assert P == 16 and S == 65
    S, P = pa.plan(1, 16, 8, 256, 16, 1025, splits=10000, sm_count=SM, kv_fp8=True)
    assert P == 32 and S == 33


def test_large_batch_plans():
    # 512 (sequence, KV head) pairs on 152 SMs: one or two splits, never more
    # (GB300, us per call for S = 1 / 2 / 3: 8K 343.8 / 338.8 / 362.9, 16K 678.8 /
    # 637.9 / 678.0; at 4K one split is 4% faster than the two the model picks)
    for L in (4096, 8192, 16384):
        S, P = pa.plan(64, 32, 8, 128, 16, L, sm_count=SM)
        assert S in (1, 2) and S * P >= L
    assert pa.plan(64, 32, 8, 128, 16, 16384, sm_count=SM)[0] == 2
    # 1024 pairs of short contexts: one split
    assert pa.plan(128, 32, 8, 128, 16, 2048, sm_count=SM)[0] == 1


def test_batch8_long_contexts():
    # 64 pairs: at 32K three full waves of seven splits beat one wave of two (GB300:
    # 166.4-169.8 vs 170.5 us); at 16K one wave of two splits, merging in their
    # clusters, is as fast or faster (86.1-86.5 vs 88.4-90.1 us for seven)
    assert pa.plan(8, 32, 8, 128, 16, 32768, sm_count=SM)[0] == 7
    assert pa.plan(8, 32, 8, 128, 16, 16384, sm_count=SM)[0] == 2
    assert pa.plan(8, 8, 8, 128, 16, 4096, sm_count=SM)[0] == 2  # 27.2 us, the best


def test_total_tokens_hint():
    # 64 sequences of 32/8 heads, mixed lengths averaging ~16.9K tokens under a 32K
    # bound: splits past each sequence's end are estimated away, so finer splits win
    # (GB300, forced splits: 752 / 715 / 709 / 692 us per call for 1 / 2 / 3 / 4)
    S0, _ = pa.plan(64, 32, 8, 128, 16, 32704, sm_count=SM)
    S1, P1 = pa.plan(64, 32, 8, 128, 16, 32704, sm_count=SM, total_tokens=64 * 16900)
    assert S0 == 2 and S1 == 4 and S1 * P1 >= 32704
    # a uniform batch's total gives the plan of no hint
    for B, Hkv, L in [(64, 8, 32768), (8, 8, 4096), (1, 4, 32768), (24, 8, 8192)]:
        assert pa.plan(B, 4 * Hkv, Hkv, 128, 16, L, sm_count=SM, total_tokens=B * L) == \
            pa.plan(B, 4 * Hkv, Hkv, 128, 16, L, sm_count=SM)
    # ignored with a window
    assert pa.plan(64, 32, 8, 128, 16, 32704, sm_count=SM, window=4096, total_tokens=64 * 1000) == \
        pa.plan(64, 32, 8, 128, 16, 32704, sm_count=SM, window=4096)


def test_many_pairs_long_context_split_in_two():
    # 512 (sequence, KV head) pairs of 32K tokens on 152 SMs: two splits shorten the
    # last of the waves (GB300: 1273 vs 1356 us per call)
    S, P = pa.plan(64, 32, 8, 128, 16, 32768, sm_count=SM)
    assert S == 2 and P == 16384


def test_kernel_count_validates_and_launches_nothing(lib):
    import torch
    n = ctypes.c_int(-1)
    # the same argument errors as the decode call, a null result, an empty batch
    assert lib.pa_decode_kernel_count(ctypes.byref(_args(Hq=12, Hkv=8)), ctypes.byref(n)) == \
        pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_kernel_count(ctypes.byref(_args(D=64)), ctypes.byref(n)) == \
        pa.PA_ERR_UNSUPPORTED
    assert lib.pa_decode_kernel_count(ctypes.byref(_args()), None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_decode_kernel_count(ctypes.byref(_args(B=0)), ctypes.byref(n)) == pa.PA_OK
    assert n.value == 0
    # pointer fields are never read: null pointers are no error here
    rc = lib.pa_decode_kernel_count(ctypes.byref(_args(q=0, k_cache=0, out=0)), ctypes.byref(n))
    if torch.cuda.is_available():
        assert rc == pa.PA_OK and n.value in (1, 2)
    else:
        assert rc == pa.PA_ERR_CUDA  # the count depends on the device

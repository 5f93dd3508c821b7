"""Python binding of libpa.so: single-query paged-attention decode on GB300.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/pa.h. PyTorch provides device
memory and the current stream. There is no CPU path: if the shared library is
missing, every call raises.

    import paged_kv_attention_pa_gb300 as pa
    out = pa.decode(q, k_cache, v_cache, block_tables, seq_lens, scale,
                    max_seq_len=4096)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

__version__ = "0.1.0"

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")

# status codes (include/pa.h)
PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA, \
    PA_ERR_OUT_OF_RANGE = range(6)
PA_F16, PA_BF16 = 0, 1
PA_KV_AS_DTYPE, PA_KV_FP8_E4M3 = 0, 1
PA_DEVERR_BLOCK_INDEX, PA_DEVERR_SEQ_LEN = 1, 2
PA_FLAG_DETERMINISTIC = 1
PA_WORKSPACE_HEADER_BYTES = 8448
PA_NOALLOC_SCRATCH_BYTES = 32 << 20
MAX_GQA_GROUP = 16

# Every symbol include/pa.h declares, with its ctypes signature.
_c = ctypes
SIGNATURES = {
    "pa_decode_workspace_bytes": (_c.c_size_t, [_c.c_int] * 5),
    "pa_decode_ex_workspace_bytes": (_c.c_size_t, [_c.c_void_p]),
    "pa_decode": (_c.c_int, [_c.c_void_p] * 6 + [_c.c_int] * 8 +
                  [_c.c_float, _c.c_int, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "pa_decode_ex": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "pa_decode_noalloc": (_c.c_int, [_c.c_void_p] * 6 + [_c.c_int] * 8 +
                          [_c.c_float, _c.c_int, _c.c_void_p]),
    "pa_decode_plan": (_c.c_int, [_c.c_void_p, _c.c_int, _c.c_void_p, _c.c_void_p]),
    "pa_decode_kernel_count": (_c.c_int, [_c.c_void_p, _c.c_void_p]),
    "pa_workspace_init": (_c.c_int, [_c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "pa_read_device_errors": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p]),
    "pa_set_device": (_c.c_int, [_c.c_int]),
    "pa_status_string": (_c.c_char_p, [_c.c_int]),
    "pa_version": (_c.c_char_p, []),
}


class DecodeArgs(ctypes.Structure):
    """Mirror of pa_decode_args (include/pa.h)."""
    _fields_ = [
        ("q", _c.c_void_p), ("k_cache", _c.c_void_p), ("v_cache", _c.c_void_p),
        ("block_tables", _c.c_void_p), ("seq_lens", _c.c_void_p), ("out", _c.c_void_p),
        ("B", _c.c_int32), ("Hq", _c.c_int32), ("Hkv", _c.c_int32), ("D", _c.c_int32),
        ("block_size", _c.c_int32), ("num_blocks", _c.c_int32),
        ("max_blocks_per_seq", _c.c_int32), ("max_seq_len", _c.c_int32),
        ("scale", _c.c_float), ("dtype", _c.c_int32), ("splits", _c.c_int32),
        ("window", _c.c_int32), ("kv_dtype", _c.c_int32),
        ("k_scale", _c.c_float), ("v_scale", _c.c_float), ("q_len", _c.c_int32),
        ("flags", _c.c_uint32), ("total_tokens", _c.c_int64),
    ]


class PAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = status_string(code) if _lib is not None else str(code)
        super().__init__(f"{where}: {msg} (status {code})")


_lib = None
_lib_lock = threading.Lock()
_tls = threading.local()


def load(path: str = LIB_PATH):
    """Load libpa.so (built in-tree). Raises if it is missing: there is no fallback."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -m paged_kv_attention_pa_gb300.build`"
                    " (the decode path has no CPU fallback)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().pa_status_string(int(code)).decode()


def version() -> str:
    return load().pa_version().decode()


_DT = {torch.float16: PA_F16, torch.bfloat16: PA_BF16}


def _ensure_device(lib, index: int):
    if getattr(_tls, "device", None) != index:
        rc = lib.pa_set_device(index)
        if rc != PA_OK:
            raise PAError(rc, "pa_set_device")
        _tls.device = index


def _stream_handle(device: torch.device, stream) -> int:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return int(s.cuda_stream)


def make_args(q, k_cache, v_cache, block_tables, seq_lens, out, scale: float,
              max_seq_len: Optional[int] = None, splits: int = 0, window: int = 0,
              k_scale: float = 1.0, v_scale: float = 1.0,
              deterministic: bool = False, total_tokens: int = 0) -> DecodeArgs:
    """Check shapes / dtypes / devices and fill a pa_decode_args. q is [B, Hq, D], or
    [B, R, Hq, D] for R causal query rows per sequence."""
    if q.dim() not in (3, 4) or k_cache.dim() != 4 or v_cache.dim() != 4:
        raise ValueError("q must be [B, Hq, D] or [B, R, Hq, D] and the caches "
                         "[num_blocks, block_size, Hkv, D]")
    if q.dim() == 4:
        B, R, Hq, D = q.shape
    else:
        (B, Hq, D), R = q.shape, 1
    nb, bs, Hkv, Dk = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or Dk != D:
        raise ValueError("k_cache / v_cache / q shapes disagree")
    fp8 = k_cache.dtype == torch.float8_e4m3fn
    if q.dtype not in _DT or out.dtype != q.dtype or v_cache.dtype != k_cache.dtype or \
            (k_cache.dtype != q.dtype and not fp8):
        raise TypeError("q and out must be float16 or bfloat16; the caches must have their "
                        "dtype or both be float8_e4m3fn")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("block_tables must be [B, max_blocks] and seq_lens [B]")
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have q's shape")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_tables", block_tables), ("seq_lens", seq_lens), ("out", out)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    a = DecodeArgs()
    a.q, a.k_cache, a.v_cache = q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr()
    a.block_tables, a.seq_lens, a.out = block_tables.data_ptr(), seq_lens.data_ptr(), out.data_ptr()
    a.B, a.Hq, a.Hkv, a.D = B, Hq, Hkv, D
    a.block_size, a.num_blocks = bs, nb
    a.max_blocks_per_seq = block_tables.shape[1]
    a.max_seq_len = 0 if max_seq_len is None else int(max_seq_len)
    a.scale = float(scale)
    a.dtype = _DT[q.dtype]
    a.splits = int(splits)
    a.window = int(window)
    a.q_len = R
    a.kv_dtype = PA_KV_FP8_E4M3 if fp8 else PA_KV_AS_DTYPE
    a.k_scale, a.v_scale = (float(k_scale), float(v_scale)) if fp8 else (1.0, 1.0)
    a.flags = PA_FLAG_DETERMINISTIC if deterministic else 0
    a.total_tokens = int(total_tokens)
    return a


# one workspace per (device, stream); grown on demand, zero-filled when made
_workspaces = {}


def workspace_for(args: DecodeArgs, device: torch.device, stream_handle: int) -> torch.Tensor:
    lib = load()
    need = lib.pa_decode_ex_workspace_bytes(ctypes.byref(args))
    if need == 0:
        raise PAError(PA_ERR_INVALID_ARG, "pa_decode_ex_workspace_bytes")
    key = (device.index, stream_handle)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
           out: Optional[torch.Tensor] = None, max_seq_len: Optional[int] = None,
           splits: int = 0, workspace: Optional[torch.Tensor] = None, stream=None,
           window: int = 0, k_scale: float = 1.0, v_scale: float = 1.0,
           deterministic: bool = False, total_tokens: int = 0) -> torch.Tensor:
    """out[b, h] = softmax(scale * q[b,h] . K_b^T) V_b over the paged context of sequence b.

    q [B, Hq, D]; k_cache, v_cache [num_blocks, block_size, Hkv, D]; block_tables
    [B, max_blocks] int32; seq_lens [B] int32; all on one CUDA device. max_seq_len
    bounds seq_lens (pass it: it sets the split plan; None means the table's
    capacity). splits > 0 forces at most that many context splits. window > 0
    attends to the last `window` tokens only. float8_e4m3fn caches are read as
    stored value * k_scale / v_scale. deterministic=True keeps fixed context splits, so
    that repeated calls are bitwise identical (by default the splits of a long context
    share out its tail as they finish, and the last bit may vary from call to call).
    total_tokens, the sum of seq_lens when the caller knows it on the host, helps the
    split plan for batches of mixed lengths. Asynchronous on the current (or given)
    stream.
    """
    lib = load()
    if out is None:
        out = torch.empty_like(q)
    args = make_args(q, k_cache, v_cache, block_tables, seq_lens, out, scale, max_seq_len, splits,
                     window, k_scale, v_scale, deterministic, total_tokens)
    _ensure_device(lib, q.device.index)
    sh = _stream_handle(q.device, stream)
    ws = workspace if workspace is not None else workspace_for(args, q.device, sh)
    rc = lib.pa_decode_ex(ctypes.byref(args), ws.data_ptr(), ws.numel(), sh)
    if rc != PA_OK:
        raise PAError(rc, "pa_decode_ex")
    return out


def decode_plain(q, k_cache, v_cache, block_tables, seq_lens, scale, out=None,
                 max_seq_len: Optional[int] = None, workspace=None, stream=None):
    """The same operation through pa_decode, the plain positional entry point."""
    lib = load()
    if out is None:
        out = torch.empty_like(q)
    args = make_args(q, k_cache, v_cache, block_tables, seq_lens, out, scale, max_seq_len, 0)
    _ensure_device(lib, q.device.index)
    sh = _stream_handle(q.device, stream)
    ws = workspace if workspace is not None else workspace_for(args, q.device, sh)
    rc = lib.pa_decode(args.q, args.k_cache, args.v_cache, args.block_tables, args.seq_lens,
                       args.out, args.B, args.Hq, args.Hkv, args.D, args.block_size,
                       args.num_blocks, args.max_blocks_per_seq, args.max_seq_len,
                       args.scale, args.dtype, ws.data_ptr(), ws.numel(), sh)
    if rc != PA_OK:
        raise PAError(rc, "pa_decode")
    return out


def decode_noalloc(q, k_cache, v_cache, block_tables, seq_lens, scale, out=None,
                   max_seq_len: Optional[int] = None, stream=None):
    """The same operation through pa_decode_noalloc: no workspace, no allocation by
    the library (the split partials live in a fixed device array of the library,
    shared by all such calls on a device; see include/pa.h for the limit)."""
    lib = load()
    if out is None:
        out = torch.empty_like(q)
    args = make_args(q, k_cache, v_cache, block_tables, seq_lens, out, scale, max_seq_len, 0)
    _ensure_device(lib, q.device.index)
    sh = _stream_handle(q.device, stream)
    rc = lib.pa_decode_noalloc(args.q, args.k_cache, args.v_cache, args.block_tables,
                               args.seq_lens, args.out, args.B, args.Hq, args.Hkv, args.D,
                               args.block_size, args.num_blocks, args.max_blocks_per_seq,
                               args.max_seq_len, args.scale, args.dtype, sh)
    if rc != PA_OK:
        raise PAError(rc, "pa_decode_noalloc")
    return out


def plan(B: int, Hq: int, Hkv: int, D: int, block_size: int, max_seq_len: int,
         splits: int = 0, sm_count: int = 0, window: int = 0,
         kv_fp8: bool = False, total_tokens: int = 0) -> Tuple[int, int]:
    """(splits, tokens per split) the library would launch with. sm_count <= 0 asks
    the current device; a positive sm_count needs no GPU. kv_fp8: FP8 E4M3 caches
    (their warp tile is 32 tokens, so splits are multiples of 32)."""
    lib = load()
    a = DecodeArgs()
    a.B, a.Hq, a.Hkv, a.D = B, Hq, Hkv, D
    a.block_size, a.num_blocks = block_size, 1
    a.max_blocks_per_seq = max(1, -(-max_seq_len // block_size))
    a.max_seq_len = max_seq_len
    a.dtype = PA_BF16
    a.splits = splits
    a.window = window
    if kv_fp8:
        a.kv_dtype, a.k_scale, a.v_scale = PA_KV_FP8_E4M3, 1.0, 1.0
    a.total_tokens = int(total_tokens)
    S, P = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib.pa_decode_plan(ctypes.byref(a), int(sm_count), ctypes.byref(S), ctypes.byref(P))
    if rc != PA_OK:
        raise PAError(rc, "pa_decode_plan")
    return S.value, P.value


def kernel_count(q, k_cache, v_cache, block_tables, seq_lens, scale, max_seq_len=None,
                 splits: int = 0, window: int = 0, total_tokens: int = 0) -> int:
    """Kernels one decode call with these tensors launches on their device (1, or 2
    with a merge grid; 0 for an empty batch). Nothing is launched."""
    lib = load()
    out = q  # only its shape and dtype are read
    args = make_args(q, k_cache, v_cache, block_tables, seq_lens, out, scale, max_seq_len,
                     splits, window, total_tokens=total_tokens)
    _ensure_device(lib, q.device.index)
    n = ctypes.c_int(-1)
    rc = lib.pa_decode_kernel_count(ctypes.byref(args), ctypes.byref(n))
    if rc != PA_OK:
        raise PAError(rc, "pa_decode_kernel_count")
    return n.value


def read_device_errors(workspace: torch.Tensor, stream=None) -> int:
    """Wait for the stream, return and clear the PA_DEVERR_* bits of a workspace."""
    lib = load()
    _ensure_device(lib, workspace.device.index)
    flags = ctypes.c_uint32(0)
    rc = lib.pa_read_device_errors(workspace.data_ptr(),
                                   _stream_handle(workspace.device, stream), ctypes.byref(flags))
    if rc != PA_OK:
        raise PAError(rc, "pa_read_device_errors")
    return flags.value


def default_workspace(device=None, stream=None) -> Optional[torch.Tensor]:
    """The workspace decode() used last on this device and stream, if any."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return _workspaces.get((dev.index, _stream_handle(dev, stream)))

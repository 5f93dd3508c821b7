"""Seeded synthetic inputs for single-query paged-attention decode.

This module is shared by the tests, the benchmark and the smoke check. It builds
inputs only: it holds none of the attention arithmetic, and neither the oracle
nor the CUDA library imports it.

What it builds, following "gqa-gate-costs-nothing" §1 (pure decode: one query
token per sequence over a fully cached context; the reference is computed from
the pre-paging K/V so that a paging bug cannot cancel itself out):

* ``q``            [B, Hq, D]                 fp16/bf16
* ``K[b], V[b]``   [L_b, Hkv, D] per sequence contiguous, pre-paging K/V
* ``k_cache``,
  ``v_cache``      [num_blocks, block_size, Hkv, D] the same rows scattered
                   into a block-paged pool through a randomly permuted table
* ``block_tables`` [B, max_blocks] int32, logical block j of sequence b lives in
                   physical block ``block_tables[b, j]``
* ``seq_lens``     [B] int32

Fills of the slots that hold no token (the unwritten tail of a sequence's last
block, and every block no table references) follow §3 and §5 of the same page:
zero, NaN in K only, NaN in V only, NaN in K and V, or finite garbage 1e4.

Draw order for a seed: seq_lens (when drawn), q, K, V, block permutation.
CPU draws use numpy's PCG64 (platform independent); CUDA draws use torch's
Philox generator and are used where the sizes make CPU generation too slow.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

POISON_MODES = ("none", "k_nan", "v_nan", "kv_nan", "kv_1e4", "kv_inf")

_DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16}
FP8 = torch.float8_e4m3fn
FP8_SCALE = 8.0 / 448.0   # default per-tensor scale: N(0,1) values to 8 sigma fit e4m3


def torch_dtype(name: str) -> torch.dtype:
    return _DTYPES[name]


@dataclass
class PagedCase:
    """One decode call's inputs, plus the contiguous K/V the oracle reads."""

    q: torch.Tensor                 # [B, Hq, D]
    K: List[torch.Tensor]           # per sequence [L_b, Hkv, D]
    V: List[torch.Tensor]
    k_cache: torch.Tensor           # [num_blocks, bs, Hkv, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor      # [B, max_blocks] int32
    seq_lens: torch.Tensor          # [B] int32
    scale: float                    # an fp32-representable value
    block_size: int
    dtype: str
    poison: str = "none"
    meta: dict = field(default_factory=dict)
    k_scale: float = 1.0            # cache element = stored value * scale (fp8 caches)
    v_scale: float = 1.0

    @property
    def kv_fp8(self) -> bool:
        return self.k_cache.dtype == FP8

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def Hq(self) -> int:
        return self.q.shape[1]

    @property
    def D(self) -> int:
        return self.q.shape[2]

    @property
    def Hkv(self) -> int:
        return self.k_cache.shape[2]

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    @property
    def max_seq_len(self) -> int:
        return int(max([int(x) for x in self.seq_lens.tolist()] + [0]))

    def to(self, device) -> "PagedCase":
        mv = lambda t: t.to(device)
        return PagedCase(mv(self.q), [mv(k) for k in self.K], [mv(v) for v in self.V],
                         mv(self.k_cache), mv(self.v_cache), mv(self.block_tables),
                         mv(self.seq_lens), self.scale, self.block_size, self.dtype,
                         self.poison, dict(self.meta), self.k_scale, self.v_scale)


def fp32_scale(D: int) -> float:
    """1/sqrt(D) rounded once to fp32; both sides of a comparison use this value."""
    return float(np.float32(1.0 / math.sqrt(D)))


def blocks_for(L: int, bs: int) -> int:
    return (L + bs - 1) // bs


def unwritten_tail_slots(L: int, bs: int) -> int:
    """Slots of the last block that hold no token: 0 when L is block-aligned."""
    return blocks_for(L, bs) * bs - L


def uniform_seq_lens(B: int, lo: int, hi: int, seed: int) -> List[int]:
    """Lengths drawn uniformly from the integers in [lo, hi] (PCG64, seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(lo, hi + 1, size=B)]


def _randn_cpu(rng: np.random.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(a).to(dtype)


def _randn_cuda(gen: torch.Generator, shape, dtype: torch.dtype, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def _fill_values(mode: str, which: str, dtype: torch.dtype) -> Optional[float]:
    """Value written into empty slots of the K ('k') or V ('v') pool, or None for zero."""
    if mode == "none":
        return None
    if mode == "k_nan":
        return float("nan") if which == "k" else None
    if mode == "v_nan":
        return float("nan") if which == "v" else None
    if mode == "kv_nan":
        return float("nan")
    if mode == "kv_1e4":
        return 1.0e4
    if mode == "kv_inf":
        return float("inf") if which == "k" else float("-inf")
    raise ValueError(f"unknown poison mode {mode!r}")


def make_case(B: int, Hq: int, Hkv: int, D: int, block_size: int,
              seq_lens: Sequence[int], dtype: str = "bf16", seed: int = 0,
              pool_factor: float = 2.0, num_blocks: Optional[int] = None,
              poison: str = "none", table_fill: str = "neg1",
              device: str = "cpu", scale: Optional[float] = None,
              max_blocks: Optional[int] = None, kv_dtype: Optional[str] = None,
              k_scale: float = FP8_SCALE, v_scale: float = FP8_SCALE) -> PagedCase:
    """Build one seeded decode call.

    ``seq_lens`` gives L_b per sequence. The pool holds ``pool_factor`` times the
    blocks the batch uses (or ``num_blocks`` when given); sequences take their
    physical blocks from one random permutation of the pool, so blocks of different
    sequences interleave. Table entries past a sequence's last block are filled with
    -1 (``table_fill='neg1'``) or with an index past the pool (``'oob'``): a correct
    kernel never reads them. ``device='cuda'`` draws on the GPU (large cases).
    ``kv_dtype='fp8'`` stores K/V as FP8 E4M3 codes of value / scale (per-tensor
    k_scale, v_scale, rounded to fp32); K[b], V[b] then hold those codes too.
    """
    assert len(seq_lens) == B
    assert Hq % Hkv == 0
    tdt = torch_dtype(dtype)
    bs = block_size
    nblk = [blocks_for(L, bs) for L in seq_lens]
    used = sum(nblk)
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(used * pool_factor)))
    assert num_blocks >= used, "pool smaller than the blocks the batch needs"
    if max_blocks is None:
        max_blocks = max(nblk + [1])

    on_cuda = str(device).startswith("cuda")
    if on_cuda:
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        rnd = lambda shape: _randn_cuda(gen, shape, tdt, device)
        perm = torch.randperm(num_blocks, generator=gen, device=device).to(torch.int64)
    else:
        rng = np.random.Generator(np.random.PCG64(seed))
        rnd = lambda shape: _randn_cpu(rng, shape, tdt)
        perm = None

    q = rnd((B, Hq, D))
    fp8 = kv_dtype == "fp8"
    k_scale = float(np.float32(k_scale)) if fp8 else 1.0
    v_scale = float(np.float32(v_scale)) if fp8 else 1.0
    if fp8:  # draw in the q dtype, then quantise value / scale to e4m3
        K = [(rnd((L, Hkv, D)).float() / k_scale).to(FP8) for L in seq_lens]
        V = [(rnd((L, Hkv, D)).float() / v_scale).to(FP8) for L in seq_lens]
        cdt = FP8
    else:
        K = [rnd((L, Hkv, D)) for L in seq_lens]
        V = [rnd((L, Hkv, D)) for L in seq_lens]
        cdt = tdt
    if perm is None:
        perm = torch.from_numpy(rng.permutation(num_blocks).astype(np.int64))

    k_cache = torch.zeros((num_blocks, bs, Hkv, D), dtype=cdt, device=device)
    v_cache = torch.zeros_like(k_cache)
    kfill = _fill_values(poison, "k", cdt)
    vfill = _fill_values(poison, "v", cdt)
    if fp8:  # e4m3 has no infinity and tops out at 448: finite garbage saturates there
        kfill = None if kfill is None else (448.0 if np.isfinite(kfill) else float("nan"))
        vfill = None if vfill is None else (448.0 if np.isfinite(vfill) else float("nan"))
    if kfill is not None:
        k_cache.fill_(kfill)
    if vfill is not None:
        v_cache.fill_(vfill)

    bad = -1 if table_fill == "neg1" else num_blocks + 7
    bt = torch.full((B, max_blocks), bad, dtype=torch.int64, device=device)
    off = 0
    for b, L in enumerate(seq_lens):
        n = nblk[b]
        bt[b, :n] = perm[off:off + n]
        off += n
        if L == 0:
            continue
        t = torch.arange(L, device=device)
        phys = bt[b, t // bs]
        slot = t % bs
        k_cache[phys, slot] = K[b]
        v_cache[phys, slot] = V[b]

    sl = torch.tensor(list(seq_lens), dtype=torch.int32, device=device)
    return PagedCase(q=q, K=K, V=V, k_cache=k_cache, v_cache=v_cache,
                     block_tables=bt.to(torch.int32), seq_lens=sl,
                     scale=fp32_scale(D) if scale is None else float(np.float32(scale)),
                     block_size=bs, dtype=dtype, poison=poison,
                     meta={"seed": seed, "num_blocks": num_blocks, "used_blocks": used},
                     k_scale=k_scale, v_scale=v_scale)


def gather_back(case: PagedCase, b: int):
    """Read sequence b's K/V back out of the pool through its block table."""
    L = int(case.seq_lens[b])
    t = torch.arange(L, device=case.k_cache.device)
    phys = case.block_tables[b, (t // case.block_size)].to(torch.int64)
    slot = t % case.block_size
    return case.k_cache[phys, slot], case.v_cache[phys, slot]


def repage(case: PagedCase, seed: int) -> PagedCase:
    """The same contiguous K/V scattered under a different random block permutation."""
    bs = case.block_size
    nb = case.num_blocks
    dev = case.k_cache.device
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = torch.from_numpy(rng.permutation(nb).astype(np.int64)).to(dev)
    k_cache = torch.empty_like(case.k_cache).copy_(case.k_cache)
    v_cache = torch.empty_like(case.v_cache).copy_(case.v_cache)
    # Empty slots keep the fill of the original pool: start from a pool filled the
    # same way, then scatter the tokens at their new homes.
    kf = _fill_values(case.poison, "k", k_cache.dtype)
    vf = _fill_values(case.poison, "v", v_cache.dtype)
    if k_cache.dtype == FP8:
        kf = None if kf is None else (448.0 if np.isfinite(kf) else float("nan"))
        vf = None if vf is None else (448.0 if np.isfinite(vf) else float("nan"))
    k_cache.fill_(0.0 if kf is None else kf)
    v_cache.fill_(0.0 if vf is None else vf)
    bt = case.block_tables.clone().to(torch.int64)
    off = 0
    for b in range(case.B):
        L = int(case.seq_lens[b])
        n = blocks_for(L, bs)
        bt[b, :n] = perm[off:off + n]
        off += n
        if L == 0:
            continue
        t = torch.arange(L, device=dev)
        k_cache[bt[b, t // bs], t % bs] = case.K[b]
        v_cache[bt[b, t // bs], t % bs] = case.V[b]
    return PagedCase(case.q, case.K, case.V, k_cache, v_cache, bt.to(torch.int32),
                     case.seq_lens, case.scale, bs, case.dtype, case.poison, dict(case.meta),
                     case.k_scale, case.v_scale)


def to_f64_numpy(t: torch.Tensor) -> np.ndarray:
    """Exact widening of an fp16/bf16 tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def fp8_codes(t: torch.Tensor) -> np.ndarray:
    """The raw uint8 codes of an FP8 E4M3 tensor (for the oracle's own decoder)."""
    return t.detach().to("cpu").view(torch.uint8).numpy()

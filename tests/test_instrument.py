"""The tail-poison harness can see the fault it is meant to catch (CPU only).

"vLLM's custom ROCm paged-attention kernel wins all sixty cells" (§3, §5 Figure 4)
insists that a clean sweep means nothing unless the instrument can see a fault:
a kernel that masks the scores past seq_len but lets the V rows of the whole final
block into the weighted sum turns NaN in the unwritten tail into NaN output
(0 * NaN = NaN), at straddling lengths only.

The mistake is planted on the CPU, in a copy of the oracle that reads through the
paged cache block by block: the "stock" arm masks scores only, the "patched" arm
also selects V rows past seq_len to zero. The same verdict the GPU tail tests use
(every output finite and rel L-inf <= 1e-2 against the float64 oracle) must flag
exactly the golden pattern: 2 dtypes x 2 GQA ratios x 4 poison modes x 2 lengths,
32 rows per arm, as in the pages' Figure 4.
"""
import numpy as np
import pytest

import pa_inputs as pi
from harness import REL_LINF_TOL, oracle_case, read_golden
from oracle import rel_linf_error


def _paged_blockwise(case, mask_v):
    """Decode through the paged cache, whole final block included (planted mistake
    when mask_v is False)."""
    bs = case.block_size
    q = pi.to_f64_numpy(case.q)
    kc = pi.to_f64_numpy(case.k_cache)
    vc = pi.to_f64_numpy(case.v_cache)
    bt = case.block_tables.numpy()
    B, Hq, D = q.shape
    Hkv = kc.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    with np.errstate(invalid="ignore"):
        for b in range(B):
            L = int(case.seq_lens[b])
            n = pi.blocks_for(L, bs)
            phys = bt[b, :n]
            Kall = kc[phys].reshape(n * bs, Hkv, D)
            Vall = vc[phys].reshape(n * bs, Hkv, D)
            live = np.arange(n * bs) < L
            for h in range(Hq):
                kv = h // G
                s = case.scale * (Kall[:, kv, :] @ q[b, h])
                s = np.where(live, s, -np.inf)           # score mask, by select
                p = np.exp(s - s[live].max())
                Vh = Vall[:, kv, :]
                if mask_v:
                    Vh = np.where(live[:, None], Vh, 0.0)  # V rows past seq_len kept out
                out[b, h] = (p @ Vh) / p.sum()
    return out


def _poisoned(y, r):
    return (not np.all(np.isfinite(y))) or rel_linf_error(y, r) > REL_LINF_TOL


GOLD = {(m, k): (int(s), int(p)) for m, k, s, p in read_golden("poison_pattern.txt")}


@pytest.mark.parametrize("mode,kind", sorted(GOLD))
def test_harness_sees_the_planted_fault(mode, kind):
    stock_hits = patched_hits = 0
    rows = 0
    for dtype in ("f16", "bf16"):
        for hq, hkv in ((16, 8), (32, 8)):
            L = 4090 if kind == "straddle" else 4096
            # narrow head_dim keeps the CPU work small; the tail arithmetic is the same
            case = pi.make_case(1, hq // 4, hkv // 4, 8, 16, [L], dtype=dtype, seed=21,
                                poison=mode)
            r = oracle_case(case)
            stock_hits += _poisoned(_paged_blockwise(case, mask_v=False), r)
            patched_hits += _poisoned(_paged_blockwise(case, mask_v=True), r)
            rows += 1
    exp_stock, exp_patched = GOLD[(mode, kind)]
    assert stock_hits == exp_stock * rows, (mode, kind, stock_hits)
    assert patched_hits == exp_patched * rows, (mode, kind, patched_hits)

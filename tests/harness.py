"""Shared test helpers: oracle on a generated case, the parity bar, golden files."""
from __future__ import annotations

import os
from typing import Iterable, Optional

import numpy as np

from oracle import decode_ref, decode_ref_one, rel_linf_error
from oracle import decode_ref_rows, dequant
from pa_inputs import PagedCase, fp8_codes, to_f64_numpy

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Relative L-infinity bar against the float64 oracle, on the reference's own
# max-abs scale ("vLLM's custom ROCm paged-attention kernel wins all sixty
# cells", §1 defines the metric; the bar is the one the decode kernel is held to).
REL_LINF_TOL = 1e-2


def read_golden(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def kv_f64(case: PagedCase, t, which: str) -> np.ndarray:
    """Contiguous K or V of one sequence as float64 cache values (fp8 decoded by the
    oracle's own E4M3 decoder and scaled)."""
    if case.kv_fp8:
        return dequant(fp8_codes(t), case.k_scale if which == "k" else case.v_scale)
    return to_f64_numpy(t)


def oracle_case(case: PagedCase, window: int = 0) -> np.ndarray:
    """Float64 oracle output for a whole case, from its contiguous K/V."""
    q = to_f64_numpy(case.q)
    K = [kv_f64(case, k, "k") for k in case.K]
    V = [kv_f64(case, v, "v") for v in case.V]
    return decode_ref(q, K, V, case.scale, window=window)


def oracle_rows(case: PagedCase, pairs: Iterable[tuple]) -> dict:
    """Oracle output for selected (b, kv_head) pairs only: {(b, kvh): [G, D]}."""
    G = case.Hq // case.Hkv
    out = {}
    for b, kvh in pairs:
        qg = to_f64_numpy(case.q[b, kvh * G:(kvh + 1) * G])
        K = kv_f64(case, case.K[b][:, kvh, :], "k")
        V = kv_f64(case, case.V[b][:, kvh, :], "v")
        out[(b, kvh)] = decode_ref_one(qg, K, V, case.scale)
    return out


# Every error assert_parity measured in this process: (what, rel L-inf error). The
# test session's summary reports the largest (tests/conftest.py).
RECORDED: list = []


def assert_parity(y: np.ndarray, r: np.ndarray, tol: float = REL_LINF_TOL, what: str = "") -> float:
    """Every output finite and max|y-r|/max|r| <= tol. Returns the error, and records it."""
    y = np.asarray(y, dtype=np.float64)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output ({int((~np.isfinite(y)).sum())} values)"
    err = rel_linf_error(y, r)
    RECORDED.append((what, float(err)))
    assert err <= tol, f"{what}: rel L-inf error {err:.3e} > {tol:.0e}"
    return err


def kv_bytes(seq_lens, Hkv: int, D: int, elem_bytes: int = 2) -> int:
    """KV bytes one decode call must read: sum_b L_b * Hkv * D * 2 (K and V) * elem."""
    return int(sum(int(L) for L in seq_lens)) * Hkv * D * 2 * elem_bytes


def oracle_rows_case(case: PagedCase) -> np.ndarray:
    """Float64 oracle for a case whose q is [B, R, Hq, D] (causal query rows)."""
    q = to_f64_numpy(case.q)
    K = [kv_f64(case, k, "k") for k in case.K]
    V = [kv_f64(case, v, "v") for v in case.V]
    return decode_ref_rows(q, K, V, case.scale)

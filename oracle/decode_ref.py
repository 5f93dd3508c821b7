"""Plain float64 single-query attention decode: the definition, written out.

Test infrastructure only (see the package docstring). Slow and obviously correct
on purpose: no blocking, no online softmax, no splitting of the context.

What it computes. "vLLM's custom ROCm paged-attention kernel wins all sixty
cells" (gqa-gate-costs-nothing), §1, fixes the problem: pure decode, one query
token per sequence and head over a fully cached context, with the reference
computed from the pre-paging K/V. For sequence b with context length L_b and
query head h, with G = Hq / Hkv query heads per KV head and the KV head of h
taken as g(h) = floor(h / G) (consecutive query heads share a KV head; the pages
do not state the mapping, this is the plainest reading of "one workgroup per
(sequence, KV head)" in "Hybrid-SSM decode rate on dual Radeon cards under vLLM",
split-KV paragraph):

    s_t        = scale * sum_d q[b, h, d] * K_b[t, g(h), d]      for t < L_b
    out[b,h,:] = sum_t softmax(s)_t * V_b[t, g(h), :]

with softmax(s)_t = exp(s_t - max s) / sum_u exp(s_u - max s), all in float64.
An empty context (L_b = 0) gives a zero row (the pages are silent; this is the
reading the tests hold the kernel to).

Error metric, same page §1: relative L-infinity against the reference's own
scale, read as  max|y - r| / max|r|  over the whole output of one call.

Parity pins: tests/test_oracle.py (brute force in 50-digit decimal arithmetic,
the float64 scaled_dot_product_attention library routine, closed forms for
equal and one-hot scores, the GQA mapping, token-order and score-shift
invariance, linearity in V, single-token contexts).
"""
from __future__ import annotations

from typing import Sequence

import numpy as np


def decode_ref_one(q_g: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Attention for the G query heads that share one KV head.

    q_g: [G, D] float64; K, V: [L, D] float64 (one KV head, contiguous tokens).
    Returns [G, D] float64. L = 0 returns zeros.
    """
    G, D = q_g.shape
    L = K.shape[0]
    if L == 0:
        return np.zeros((G, V.shape[1] if V.ndim == 2 else D), dtype=np.float64)
    s = float(scale) * (q_g @ K.T)                  # [G, L] scores
    s_max = s.max(axis=1, keepdims=True)            # per head, over tokens
    e = np.exp(s - s_max)
    w = e / e.sum(axis=1, keepdims=True)            # softmax over tokens
    return w @ V                                     # [G, D]


def decode_ref(q: np.ndarray, K_list: Sequence[np.ndarray], V_list: Sequence[np.ndarray],
               scale: float, window: int = 0) -> np.ndarray:
    """Decode for a whole batch.

    q: [B, Hq, D] float64. K_list[b], V_list[b]: [L_b, Hkv, D] float64, the
    contiguous (pre-paging) keys and values of sequence b. scale: the fp32 scale
    widened to float64. window > 0 restricts every query to the last `window`
    tokens of its context, t in [max(0, L_b - window), L_b): the sliding-window
    layers of "vLLM's custom ROCm paged-attention kernel wins all sixty cells" (§4:
    a sliding layer scans 1024 tokens while a full layer scans the whole context).
    window <= 0 is the full context. Returns out [B, Hq, D] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        K = np.asarray(K_list[b], dtype=np.float64)
        V = np.asarray(V_list[b], dtype=np.float64)
        if window > 0:
            lo = max(0, K.shape[0] - window)
            K, V = K[lo:], V[lo:]
        if K.shape[0] == 0:
            continue
        Hkv = K.shape[1]
        assert Hq % Hkv == 0, "query heads must be a multiple of KV heads"
        G = Hq // Hkv
        for kvh in range(Hkv):
            heads = slice(kvh * G, (kvh + 1) * G)
            out[b, heads, :] = decode_ref_one(q[b, heads, :], K[:, kvh, :], V[:, kvh, :], scale)
    return out


def rel_linf_error(y: np.ndarray, r: np.ndarray) -> float:
    """max|y - r| / max|r| (falls back to max|y - r| when r is all zero).

    Any non-finite y gives +inf, so a NaN or Inf output can never pass a bound.
    """
    y = np.asarray(y, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if not np.all(np.isfinite(y)):
        return float("inf")
    num = float(np.max(np.abs(y - r))) if y.size else 0.0
    den = float(np.max(np.abs(r))) if r.size else 0.0
    return num / den if den > 0.0 else num


def decode_ref_rows(q: np.ndarray, K_list: Sequence[np.ndarray], V_list: Sequence[np.ndarray],
                    scale: float) -> np.ndarray:
    """Decode with several query rows per sequence, causal among the new rows.

    q: [B, R, Hq, D] float64: the queries of the last R tokens of each context
    (speculative-decode rows, or the tail of a chunked prefill; "vLLM's custom ROCm
    paged-attention kernel wins all sixty cells", §6, names speculation that makes
    decode carry several query rows). Row i of sequence b is the query of token
    L_b - R + i and attends to the tokens t < L_b - R + i + 1: every earlier token
    and itself. A row left with no tokens (L_b < R - i) gives zeros. Each row is
    the single-row definition over its own prefix of K/V. Returns [B, R, Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    B, R, Hq, D = q.shape
    out = np.zeros((B, R, Hq, D), dtype=np.float64)
    for b in range(B):
        K = np.asarray(K_list[b], dtype=np.float64)
        V = np.asarray(V_list[b], dtype=np.float64)
        L = K.shape[0]
        for i in range(R):
            lim = L - R + i + 1
            if lim <= 0:
                continue
            out[b, i] = decode_ref(q[b, i][None], [K[:lim]], [V[:lim]], scale)[0]
    return out

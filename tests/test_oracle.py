"""Pins for the float64 oracle, each independent of the oracle's own code.

Every pin is written against something the oracle does not contain: 50-digit
decimal brute force, torch's float64 scaled_dot_product_attention, closed forms
(equal scores give the mean of V, a one-hot score selects one V row, a single
token returns its V row, a GQA head reads its own KV head), and invariances of
softmax attention (token order, a common score shift, linearity in V).

The mutant section plants plausible mistakes in copies of the oracle and checks
that at least one pin fails for each, so the pins are known to bite.
"""
import decimal
import math

import numpy as np
import pytest
import torch

from oracle import decode_ref, rel_linf_error

pytestmark = []


# ----------------------------------------------------------------- helpers
def _rand_problem(seed, B=2, Hq=4, Hkv=2, D=4, lens=(3, 8), scale=0.5):
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((B, Hq, D))
    K = [rng.standard_normal((L, Hkv, D)) for L in lens]
    V = [rng.standard_normal((L, Hkv, D)) for L in lens]
    return q, K, V, scale


def _brute_force_decimal(q, K, V, scale, digits=50):
    """exp(s)/sum exp(s) with no max subtraction, in 50-digit decimal arithmetic."""
    ctx = decimal.Context(prec=digits)
    Dd = lambda x: ctx.create_decimal(repr(float(x)))
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = K[b].shape[0]
        Hkv = K[b].shape[1]
        G = Hq // Hkv
        for h in range(Hq):
            kv = h // G
            s = []
            for t in range(L):
                acc = ctx.create_decimal(0)
                for d in range(D):
                    acc = ctx.add(acc, ctx.multiply(Dd(q[b, h, d]), Dd(K[b][t, kv, d])))
                s.append(ctx.multiply(Dd(scale), acc))
            e = [ctx.exp(x) for x in s]
            z = sum(e, ctx.create_decimal(0))
            for d in range(D):
                num = sum((ctx.multiply(e[t], Dd(V[b][t, kv, d])) for t in range(L)),
                          ctx.create_decimal(0))
                out[b, h, d] = float(ctx.divide(num, z)) if L else 0.0
    return out


def _sdpa_f64(q, K, V, scale):
    """torch's float64 scaled_dot_product_attention, GQA by repeat_interleave."""
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D))
    for b in range(B):
        Hkv = K[b].shape[1]
        G = Hq // Hkv
        qt = torch.from_numpy(q[b]).unsqueeze(1)                       # [Hq, 1, D]
        kt = torch.from_numpy(K[b]).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, L, D]
        vt = torch.from_numpy(V[b]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        out[b] = o[:, 0, :].numpy()
    return out


# Each pin takes the decode function under test and raises AssertionError on failure.
def pin_brute_force(fn):
    for seed, lens in [(1, (1, 3)), (2, (8, 5)), (3, (2, 7))]:
        q, K, V, scale = _rand_problem(seed, lens=lens)
        r = _brute_force_decimal(q, K, V, scale)
        y = fn(q, K, V, scale)
        assert np.allclose(y, r, rtol=0, atol=1e-14 * max(1.0, np.abs(r).max())), \
            f"brute force mismatch {np.abs(y - r).max()}"


def pin_sdpa(fn):
    for seed in (4, 5):
        q, K, V, scale = _rand_problem(seed, B=2, Hq=6, Hkv=2, D=16, lens=(33, 17), scale=0.25)
        r = _sdpa_f64(q, K, V, scale)
        y = fn(q, K, V, scale)
        assert np.abs(y - r).max() <= 1e-12 * np.abs(r).max(), "sdpa float64 mismatch"


def pin_equal_scores_mean(fn):
    q, K, V, scale = _rand_problem(6, lens=(5, 9))
    q = np.zeros_like(q)
    y = fn(q, K, V, scale)
    for b in range(q.shape[0]):
        G = q.shape[1] // K[b].shape[1]
        for h in range(q.shape[1]):
            expect = V[b][:, h // G, :].mean(axis=0)
            assert np.abs(y[b, h] - expect).max() <= 1e-15 * max(1, np.abs(expect).max()) * 8, \
                "q=0 must give the mean of V"


def pin_one_hot(fn):
    rng = np.random.Generator(np.random.PCG64(7))
    D, L, t0, c = 8, 6, 4, 1.0e3
    qv = rng.standard_normal(D)
    # K rows orthogonal to q except row t0, whose score is exactly c (scale 1).
    K = rng.standard_normal((L, 1, D))
    for t in range(L):
        K[t, 0] -= (K[t, 0] @ qv) / (qv @ qv) * qv
    K[t0, 0] = c * qv / (qv @ qv)
    V = rng.standard_normal((L, 1, D))
    y = fn(qv.reshape(1, 1, D), [K], [V], 1.0)
    assert np.abs(y[0, 0] - V[t0, 0]).max() <= 1e-12, "one-hot score must select V[t0]"


def pin_single_token(fn):
    q, K, V, scale = _rand_problem(8, lens=(1, 1))
    y = fn(q, K, V, scale)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(y[b, h], V[b][0, h // 2]), "L=1 must return V[0]"


def pin_gqa_mapping(fn):
    rng = np.random.Generator(np.random.PCG64(9))
    B, Hq, Hkv, D, L = 1, 12, 4, 4, 7
    q = rng.standard_normal((B, Hq, D))
    K = [rng.standard_normal((L, Hkv, D))]
    V = [np.zeros((L, Hkv, D))]
    for k in range(Hkv):
        V[0][:, k, :] = float(k)
    y = fn(q, K, V, 0.3)
    for h in range(Hq):
        assert np.allclose(y[0, h], h // (Hq // Hkv), rtol=0, atol=1e-14), \
            f"head {h} must read KV head {h // (Hq // Hkv)}"


def pin_token_order(fn):
    q, K, V, scale = _rand_problem(10, lens=(11, 6))
    y = fn(q, K, V, scale)
    rng = np.random.Generator(np.random.PCG64(11))
    Kp, Vp = [], []
    for k, v in zip(K, V):
        p = rng.permutation(k.shape[0])
        Kp.append(k[p])
        Vp.append(v[p])
    y2 = fn(q, Kp, Vp, scale)
    assert np.abs(y - y2).max() <= 1e-14 * np.abs(y).max() * 4, "K/V rows must move together"


def pin_score_shift(fn):
    # Adding lam * q_h/|q_h|^2 to every K row of a head shifts all its scores by the
    # same scale*lam: softmax is unchanged. One head per KV head so the shift is exact.
    rng = np.random.Generator(np.random.PCG64(12))
    B, Hq, D, L = 1, 3, 5, 9
    q = rng.standard_normal((B, Hq, D))
    K = [rng.standard_normal((L, Hq, D))]
    V = [rng.standard_normal((L, Hq, D))]
    y = fn(q, K, V, 0.7)
    Ks = K[0].copy()
    for h in range(Hq):
        Ks[:, h, :] += 40.0 * q[0, h] / (q[0, h] @ q[0, h])
    y2 = fn(q, [Ks], V, 0.7)
    assert np.abs(y - y2).max() <= 1e-11 * np.abs(y).max(), "a common score shift must not matter"


def pin_linear_in_v(fn):
    q, K, V, scale = _rand_problem(13, lens=(6, 4))
    _, _, W, _ = _rand_problem(14, lens=(6, 4))
    y1 = fn(q, K, V, scale)
    y2 = fn(q, K, W, scale)
    y3 = fn(q, K, [a + 2.0 * b for a, b in zip(V, W)], scale)
    assert np.abs(y3 - (y1 + 2.0 * y2)).max() <= 1e-13 * np.abs(y3).max() * 4, "output is linear in V"


def pin_two_token_closed_form(fn):
    # Two tokens with scores a, b: weights 1/(1+e^(b-a)) and 1/(1+e^(a-b)).
    D = 3
    q = np.array([[[1.0, 2.0, -1.0]]])
    K = [np.array([[[0.5, 0.0, 0.0]], [[0.0, 0.0, 2.0]]])]   # q.k = 0.5, -2.0
    V = [np.array([[[1.0, 0.0, 3.0]], [[0.0, 1.0, -1.0]]])]
    scale = 0.8
    a, b = scale * 0.5, scale * -2.0
    w0 = 1.0 / (1.0 + math.exp(b - a))
    w1 = 1.0 / (1.0 + math.exp(a - b))
    expect = w0 * V[0][0, 0] + w1 * V[0][1, 0]
    y = fn(q, K, V, scale)
    assert np.abs(y[0, 0] - expect).max() <= 1e-15 * 4, "two-token closed form"


def pin_empty_context(fn):
    q, K, V, scale = _rand_problem(15, lens=(0, 3))
    y = fn(q, K, V, scale)
    assert np.all(y[0] == 0.0), "an empty context gives a zero row"
    assert np.all(np.isfinite(y))


PINS = [pin_brute_force, pin_sdpa, pin_equal_scores_mean, pin_one_hot, pin_single_token,
        pin_gqa_mapping, pin_token_order, pin_score_shift, pin_linear_in_v,
        pin_two_token_closed_form, pin_empty_context]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(decode_ref)


# ----------------------------------------------------------------- mutants
def _make_mutant(kind):
    def fn(q, K_list, V_list, scale):
        B, Hq, D = q.shape
        out = np.zeros((B, Hq, D))
        for b in range(B):
            K, V = K_list[b], V_list[b]
            L = K.shape[0]
            if L == 0:
                if kind == "empty_nan":
                    out[b] = np.nan
                continue
            Hkv = K.shape[1]
            G = Hq // Hkv
            for h in range(Hq):
                kv = (h % Hkv) if kind == "gqa_mod" else h // G
                sc = 1.0 if kind == "no_scale" else scale
                s = sc * (K[:, kv, :] @ q[b, h])
                if kind == "drop_last":
                    s, Vv = s[:-1], V[:-1, kv, :]
                else:
                    Vv = V[:, kv, :]
                if kind == "no_max_sub":
                    e = np.exp(s)
                elif kind == "sign":
                    e = np.exp(-(s - s.min()))
                else:
                    e = np.exp(s - s.max())
                w = e / e.sum()
                if kind == "kv_swap":
                    out[b, h] = w @ K[:, kv, :]
                elif kind == "v_shift":
                    out[b, h] = w @ np.roll(Vv, 1, axis=0)
                elif kind == "no_norm":
                    out[b, h] = e @ Vv
                else:
                    out[b, h] = w @ Vv
        return out
    return fn


MUTANTS = ["gqa_mod", "no_scale", "drop_last", "no_max_sub", "sign", "kv_swap",
           "v_shift", "no_norm", "empty_nan"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_mutant(kind):
    fn = _make_mutant(kind)
    failed = []
    with np.errstate(all="ignore"):
        for pin in PINS:
            try:
                pin(fn)
            except (AssertionError, FloatingPointError, ValueError, IndexError):
                failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {kind!r}"


def test_unmutated_copy_passes_all_pins():
    fn = _make_mutant("none")
    for pin in PINS:
        pin(fn)


# ----------------------------------------------------------------- error metric
def test_rel_linf_error():
    r = np.array([[1.0, -4.0], [2.0, 0.5]])
    y = r.copy()
    y[0, 1] += 0.04
    assert rel_linf_error(y, r) == pytest.approx(0.01)
    y[1, 0] = np.nan
    assert rel_linf_error(y, r) == float("inf")
    assert rel_linf_error(np.zeros(3), np.zeros(3)) == 0.0


# ----------------------------------------------------------------- sliding window
def test_window_at_least_context_is_full_decode():
    q, K, V, scale = _rand_problem(40, lens=(9, 5))
    full = decode_ref(q, K, V, scale)
    assert np.array_equal(decode_ref(q, K, V, scale, window=9), full)
    assert np.array_equal(decode_ref(q, K, V, scale, window=100), full)
    assert np.array_equal(decode_ref(q, K, V, scale, window=0), full)


def test_window_one_returns_last_value_row():
    q, K, V, scale = _rand_problem(41, lens=(9, 5))
    y = decode_ref(q, K, V, scale, window=1)
    for b, L in enumerate((9, 5)):
        for h in range(4):
            assert np.array_equal(y[b, h], V[b][L - 1, h // 2])


def test_window_brute_force():
    # the window is the last W tokens: brute force over exactly those tokens
    q, K, V, scale = _rand_problem(42, lens=(8, 3))
    W = 3
    y = decode_ref(q, K, V, scale, window=W)
    r = _brute_force_decimal(q, [k[-W:] for k in K], [v[-W:] for v in V], scale)
    assert np.abs(y - r).max() <= 1e-14 * max(1.0, np.abs(r).max())


def test_window_pins_catch_off_by_one():
    # a plausible mistake (window starting one token late) fails the brute force pin
    q, K, V, scale = _rand_problem(43, lens=(8, 6))
    W = 4
    wrong = decode_ref(q, [k[1:] for k in K], [v[1:] for v in V], scale, window=W - 1)
    r = _brute_force_decimal(q, [k[-W:] for k in K], [v[-W:] for v in V], scale)
    assert np.abs(wrong - r).max() > 1e-6


# ----------------------------------------------------------------- several query rows
from oracle import decode_ref_rows


def test_rows_one_row_is_decode():
    q, K, V, scale = _rand_problem(44, lens=(7, 3))
    y = decode_ref_rows(q[:, None], K, V, scale)
    assert np.array_equal(y[:, 0], decode_ref(q, K, V, scale))


def test_rows_brute_force_causal():
    # brute force each row over exactly the tokens up to its own position
    rng = np.random.Generator(np.random.PCG64(45))
    B, R, Hq, Hkv, D = 2, 3, 4, 2, 4
    lens = (6, 4)
    q = rng.standard_normal((B, R, Hq, D))
    K = [rng.standard_normal((L, Hkv, D)) for L in lens]
    V = [rng.standard_normal((L, Hkv, D)) for L in lens]
    y = decode_ref_rows(q, K, V, 0.5)
    for b, L in enumerate(lens):
        for i in range(R):
            lim = L - R + i + 1
            r = _brute_force_decimal(q[b, i][None], [K[b][:lim]], [V[b][:lim]], 0.5)
            assert np.abs(y[b, i] - r[0]).max() <= 1e-14 * max(1.0, np.abs(r).max())


def test_rows_causality():
    # changing token t only changes the rows that can see it
    rng = np.random.Generator(np.random.PCG64(46))
    B, R, L = 1, 4, 9
    q = rng.standard_normal((B, R, 2, 4))
    K = [rng.standard_normal((L, 1, 4))]
    V = [rng.standard_normal((L, 1, 4))]
    y = decode_ref_rows(q, K, V, 0.7)
    t = L - 2                      # visible to rows 2 and 3 only
    K2 = [K[0].copy()]
    V2 = [V[0].copy()]
    K2[0][t] += 3.0
    V2[0][t] -= 5.0
    y2 = decode_ref_rows(q, K2, V2, 0.7)
    assert np.array_equal(y[0, :2], y2[0, :2])
    assert np.abs(y[0, 2:] - y2[0, 2:]).min() > 0


def test_rows_short_context_gives_zero_rows():
    rng = np.random.Generator(np.random.PCG64(47))
    q = rng.standard_normal((1, 4, 2, 4))
    K = [rng.standard_normal((2, 1, 4))]
    V = [rng.standard_normal((2, 1, 4))]
    y = decode_ref_rows(q, K, V, 1.0)
    assert np.all(y[0, :2] == 0) and np.all(np.isfinite(y))
    assert np.array_equal(y[0, 2, 0], V[0][0, 0])   # row 2 sees one token

"""CUDA path against the float64 oracle, through the C ABI (GB300 only).

Bar: every output finite and rel L-inf <= 1e-2 against the oracle on the
reference's own max-abs scale ("vLLM's custom ROCm paged-attention kernel wins
all sixty cells", §1). Small cases compare every output; full-size cases compare
sampled (sequence, KV head) groups the oracle computes one by one. Inputs are the
seeded synthetic shapes of the pages' sweeps (§1-§3 of that page; the hybrid
layer of "Hybrid-SSM decode rate on dual Radeon cards under vLLM").
"""
import random

import numpy as np
import pytest
import torch

import pa_inputs as pi
from harness import (REL_LINF_TOL, assert_parity, oracle_case, oracle_rows, oracle_rows_case,
                     read_golden)

pytestmark = pytest.mark.gpu

GRID_SHAPES = [(8, 8), (16, 8), (24, 8), (32, 8), (32, 16)]


def run(pa, case, **kw):
    c = case if case.q.is_cuda else case.to("cuda")
    if c.kv_fp8:
        kw.setdefault("k_scale", c.k_scale)
        kw.setdefault("v_scale", c.v_scale)
    out = pa.decode(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, c.scale,
                    max_seq_len=kw.pop("max_seq_len", c.max_seq_len), **kw)
    torch.cuda.synchronize()
    return out


def no_device_errors(pa):
    ws = pa.default_workspace()
    assert ws is not None
    assert pa.read_device_errors(ws) == 0


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_diff(a, b):
    """max |a - b| / max |b|: how far two outputs of the same call drift apart."""
    a, b = to_np(a), to_np(b)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


# Two outputs of one call whose splits group the tokens differently (the splits of a
# long context share out its tail tile by tile) differ by more than fp32 summation
# order: each warp rounds its softmax weights to the MMA type relative to its own
# running maximum, which depends on the tokens it streamed. That is the rounding the
# error band of "vLLM's custom ROCm paged-attention kernel wins all sixty cells"
# (§3) already contains, so two such outputs are held to the parity bar of each
# other; each is also checked against the oracle, and the exact tile-count test
# catches a token counted twice or skipped.
ORDER_TOL = REL_LINF_TOL


def check_sampled(pa, case, out, pairs, what):
    ref = oracle_rows(case, pairs)
    G = case.Hq // case.Hkv
    errs = []
    for (b, kvh), r in ref.items():
        y = to_np(out[b, kvh * G:(kvh + 1) * G])
        errs.append(assert_parity(y, r, what=f"{what} b={b} kvh={kvh}"))
    return max(errs)


# ------------------------------------------------------------------ smoke config
def test_first_config(cuda_lib):
    # batch 1, 8/8 heads, head_dim 128, block 16, seq 512, 32 blocks of a 64-block cache
    case = pi.make_case(1, 8, 8, 128, 16, [512], seed=0, num_blocks=64)
    y = run(cuda_lib, case)
    err = assert_parity(to_np(y), oracle_case(case), what="first config")
    assert err < 5e-3
    no_device_errors(cuda_lib)


def test_plain_and_ex_entry_points_agree(cuda_lib):
    case = pi.make_case(2, 16, 8, 128, 16, [700, 1500], seed=1).to("cuda")
    a = run(cuda_lib, case)
    b = cuda_lib.decode_plain(case.q, case.k_cache, case.v_cache, case.block_tables,
                              case.seq_lens, case.scale, max_seq_len=case.max_seq_len)
    torch.cuda.synchronize()
    assert rel_diff(a, b) <= ORDER_TOL


# ------------------------------------------------------------------ GQA x depth grid
@pytest.mark.parametrize("hq,hkv", GRID_SHAPES)
@pytest.mark.parametrize("B", [1, 8])
def test_grid_small_full_compare(cuda_lib, hq, hkv, B):
    # every output compared, at depths the oracle finishes quickly
    for L in (1024, 2048):
        case = pi.make_case(B, hq, hkv, 128, 16, [L] * B, seed=L + B)
        y = run(cuda_lib, case)
        assert_parity(to_np(y), oracle_case(case), what=f"grid {hq}/{hkv} B={B} L={L}")
    no_device_errors(cuda_lib)


@pytest.mark.parametrize("hq,hkv", GRID_SHAPES)
def test_grid_full_depths_sampled(cuda_lib, hq, hkv):
    rng = random.Random(hq * 100 + hkv)
    for B in (1, 8):
        for L in (4096, 8192, 16384, 32768):
            case = pi.make_case(B, hq, hkv, 128, 16, [L] * B, seed=7, device="cuda")
            y = run(cuda_lib, case)
            pairs = {(rng.randrange(B), rng.randrange(hkv)) for _ in range(3)}
            check_sampled(cuda_lib, case, y, sorted(pairs), f"grid {hq}/{hkv} B={B} L={L}")
            assert torch.isfinite(y).all()
            del case, y
    no_device_errors(cuda_lib)


# ------------------------------------------------------------------ tail straddle
TAIL_LENS = [1023, 1025, 4095, 4097, 16385, 1024, 4096]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8)])
@pytest.mark.parametrize("L", TAIL_LENS)
def test_tail_poison_matrix(cuda_lib, dtype, hq, hkv, L):
    outs = {}
    for mode in pi.POISON_MODES:
        case = pi.make_case(1, hq, hkv, 128, 16, [L], dtype=dtype, seed=3, poison=mode)
        y = run(cuda_lib, case)
        if mode == "none":
            ref = oracle_case(case)
        assert_parity(to_np(y), ref, what=f"tail {mode} L={L} {dtype} {hq}/{hkv}")
        outs[mode] = run(cuda_lib, case, deterministic=True)
    # the fill of the empty slots must not change a single bit of the output
    for mode, y in outs.items():
        assert torch.equal(y, outs["none"]), f"output depends on the {mode} fill"
    no_device_errors(cuda_lib)


def test_tail_batch_of_all_lengths(cuda_lib):
    lens = [1023, 1025, 4095, 4097, 16385]
    for mode in ("v_nan", "kv_nan", "kv_1e4"):
        case = pi.make_case(5, 32, 8, 128, 16, lens, seed=4, poison=mode)
        y = run(cuda_lib, case)
        assert_parity(to_np(y), oracle_case(case), what=f"tail batch {mode}")


def test_poison_pattern_golden_on_gpu(cuda_lib):
    # The patched column of the pages' Figure 4: no mode poisons at any length.
    for mode, kind, stock, patched in read_golden("poison_pattern.txt"):
        L = 4090 if kind == "straddle" else 4096
        case = pi.make_case(1, 16, 8, 128, 16, [L], seed=5, poison=mode)
        y = run(cuda_lib, case)
        poisoned = (not torch.isfinite(y).all().item())
        assert int(poisoned) == int(patched) == 0


# ------------------------------------------------------------------ hybrid layer
@pytest.mark.parametrize("L", [500, 1000, 2048, 4096, 8192, 12288, 16384, 20480, 24576,
                               28672, 32768])
def test_hybrid_layer(cuda_lib, L):
    # 24 query / 4 KV heads (ratio 6), head_dim 256, block 784 (non power of two)
    case = pi.make_case(1, 24, 4, 256, 784, [L], seed=L)
    y = run(cuda_lib, case)
    assert_parity(to_np(y), oracle_case(case), what=f"hybrid L={L}")
    no_device_errors(cuda_lib)


@pytest.mark.parametrize("L", [4096, 32768])
def test_hybrid_step_graph_of_16_layers(cuda_lib, L):
    # One decode step of the hybrid model's full-attention layers: 16 independent
    # layer calls, each on its own cache and block table ("Hybrid-SSM decode rate on
    # dual Radeon cards under vLLM", profile paragraph: 16 calls per step), captured
    # as one CUDA graph and replayed; every layer's output against the oracle.
    layers = [pi.make_case(1, 24, 4, 256, 784, [L], seed=160 + i, device="cuda",
                           poison="kv_nan" if i % 2 else "none") for i in range(16)]
    outs = [torch.empty_like(c.q) for c in layers]
    s = torch.cuda.Stream()

    def step():
        for c, o in zip(layers, outs):
            cuda_lib.decode(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, c.scale,
                            out=o, max_seq_len=L, stream=s)

    with torch.cuda.stream(s):
        step()  # sizes the stream's workspace before the capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
    for rep in range(2):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for i, (c, o) in enumerate(zip(layers, outs)):
            assert_parity(to_np(o), oracle_case(c), what=f"step L={L} layer {i} replay {rep}")
    ws = cuda_lib.default_workspace(layers[0].q.device, s)
    assert ws is not None and cuda_lib.read_device_errors(ws, stream=s) == 0


def test_hybrid_nan_spare(cuda_lib):
    case = pi.make_case(1, 24, 4, 256, 784, [5000], seed=8, poison="kv_nan")
    ref = oracle_case(case)
    y = run(cuda_lib, case)
    assert_parity(to_np(y), ref, what="hybrid nan spare")
    clean = pi.make_case(1, 24, 4, 256, 784, [5000], seed=8, poison="none")
    assert torch.equal(run(cuda_lib, case, deterministic=True),
                       run(cuda_lib, clean, deterministic=True))


# ------------------------------------------------------------------ mixed serving batch
def test_mixed_serving_batch(cuda_lib):
    lens = pi.uniform_seq_lens(64, 1024, 32768, seed=0)
    case = pi.make_case(64, 32, 8, 128, 16, lens, seed=0, pool_factor=1.1, poison="kv_nan",
                        device="cuda")
    y = run(cuda_lib, case)
    assert torch.isfinite(y).all()
    rng = random.Random(0)
    pairs = sorted({(rng.randrange(64), rng.randrange(8)) for _ in range(12)} |
                   {(int(np.argmax(lens)), 0), (int(np.argmin(lens)), 7)})
    check_sampled(cuda_lib, case, y, pairs, "mixed batch")
    no_device_errors(cuda_lib)


# ------------------------------------------------------------------ error margin
# The parity bar is 1e-2; the pages observed 2.12e-3 .. 4.72e-3 for bf16 against
# their reference ("vLLM's custom ROCm paged-attention kernel wins all sixty cells",
# Abstract and Figure 2). The bar alone would let the error drift to twice that band
# unnoticed, so the largest error over one fixed case of every workload (C1 .. C5)
# is held to ERROR_BAND. For bf16 the band sits one quarter above the pages' upper
# figure: the kernel rounds the softmax weights to the MMA type once per tile (bf16
# carries 8 significant bits, a relative rounding of up to 2^-9 per weight) and the
# output once, the same roundings as a bf16 kernel of the pages. fp16 makes the
# same roundings with 11 significant bits (8 times finer): its band is an eighth of
# the pages' figure with a factor of two of margin.
ERROR_BAND = {"bf16": 6e-3, "f16": 1.5e-3}


def margin_cases(dtype):
    """(name, case, pairs): pairs None = compare every output, else sampled groups."""
    yield "C1", pi.make_case(1, 8, 8, 128, 16, [512], dtype=dtype, seed=0, num_blocks=64), None
    for i, (hq, hkv) in enumerate(GRID_SHAPES):
        yield (f"C2 {hq}/{hkv} B=8 L=2048",
               pi.make_case(8, hq, hkv, 128, 16, [2048] * 8, dtype=dtype, seed=140 + i), None)
    yield ("C2 8/8 B=1 L=32768",
           pi.make_case(1, 8, 8, 128, 16, [32768], dtype=dtype, seed=146, device="cuda"),
           [(0, 0), (0, 5)])
    yield ("C3 32/8 L=4097 kv_nan",
           pi.make_case(1, 32, 8, 128, 16, [4097], dtype=dtype, seed=147, poison="kv_nan"), None)
    yield ("C3 16/8 L=16385 v_nan",
           pi.make_case(1, 16, 8, 128, 16, [16385], dtype=dtype, seed=148, poison="v_nan"), None)
    for L in (4096, 32768):
        yield (f"C4 hybrid L={L}",
               pi.make_case(1, 24, 4, 256, 784, [L], dtype=dtype, seed=149 + L), None)
    lens = pi.uniform_seq_lens(64, 1024, 32768, seed=0)
    yield ("C5 mixed",
           pi.make_case(64, 32, 8, 128, 16, lens, dtype=dtype, seed=0, pool_factor=1.1,
                        poison="kv_nan", device="cuda"),
           [(int(np.argmax(lens)), 0), (int(np.argmin(lens)), 7), (17, 3), (40, 5)])


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_error_stays_in_band(cuda_lib, dtype):
    errs = {}
    for name, case, pairs in margin_cases(dtype):
        y = run(cuda_lib, case)
        if pairs is None:
            errs[name] = assert_parity(to_np(y), oracle_case(case), what=f"{name} {dtype}")
        else:
            errs[name] = check_sampled(cuda_lib, case, y, pairs, f"{name} {dtype}")
        del case, y
    worst = max(errs, key=errs.get)
    print(f"largest rel L-inf error ({dtype}): {errs[worst]:.3e} in {worst}; " +
          ", ".join(f"{k} {v:.2e}" for k, v in errs.items()))
    band = ERROR_BAND[dtype]
    assert errs[worst] <= band, f"{worst}: {errs[worst]:.3e} outside the {band} band"


def test_grouping_spread(cuda_lib):
    # Outputs of one call under different groupings of its tokens (split counts, fixed
    # or shared tails) against each other: each is within the band of the oracle, so
    # two differ by at most twice the band; report and hold the largest difference.
    spread = 0.0
    for case in (pi.make_case(2, 24, 8, 128, 16, [4097, 1365], seed=150).to("cuda"),
                 pi.make_case(1, 24, 4, 256, 784, [32768], seed=151, device="cuda"),
                 pi.make_case(1, 8, 8, 128, 16, [32768], seed=152, device="cuda")):
        outs = [run(cuda_lib, case, splits=S, deterministic=det)
                for S in (0, 1, 2, 3, 7) for det in (False, True)]
        for i in range(len(outs)):
            for j in range(i):
                spread = max(spread, rel_diff(outs[i], outs[j]))
    print(f"largest difference between groupings of one call: {spread:.3e}")
    assert spread <= ORDER_TOL


# ------------------------------------------------------------------ splits
@pytest.mark.parametrize("L", [1025, 4097])
def test_split_sweep(cuda_lib, L):
    case = pi.make_case(2, 24, 8, 128, 16, [L, L // 3], seed=9).to("cuda")
    ref = oracle_case(case)
    results = {}
    for S in (1, 2, 3, 7, 10000):
        y = run(cuda_lib, case, splits=S)
        assert_parity(to_np(y), ref, what=f"splits={S} L={L}")
        yd = run(cuda_lib, case, splits=S, deterministic=True)
        assert_parity(to_np(yd), ref, what=f"splits={S} L={L} deterministic")
        y2 = run(cuda_lib, case, splits=S, deterministic=True)
        assert torch.equal(yd, y2), "fixed splits must give bit-identical results"
        assert rel_diff(y, yd) <= ORDER_TOL
        results[S] = y
    no_device_errors(cuda_lib)


def test_split_sweep_head256(cuda_lib):
    case = pi.make_case(1, 24, 4, 256, 784, [3000], seed=10).to("cuda")
    ref = oracle_case(case)
    for S in (1, 2, 5, 94):
        assert_parity(to_np(run(cuda_lib, case, splits=S)), ref, what=f"d256 splits={S}")


def test_workspace_reused_across_shapes(cuda_lib):
    # one workspace, calls of different (B, Hkv, splits) in a row: each call must
    # find its counters at zero whatever the previous call stored in the partials
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    for B, hq, hkv, L in [(8, 32, 8, 1024), (8, 32, 16, 1024), (2, 64, 64, 2500),
                          (1, 24, 4, 3000), (8, 32, 16, 4096)]:
        D = 256 if hkv == 4 else 128
        bs = 784 if hkv == 4 else 16
        case = pi.make_case(B, hq, hkv, D, bs, [L] * B, seed=B + hkv)
        y = run(cuda_lib, case, workspace=ws)
        assert_parity(to_np(y), oracle_case(case), what=f"reuse {B}x{hq}/{hkv} L={L}")
        assert cuda_lib.read_device_errors(ws) == 0


# ------------------------------------------------------------------ shared tiles
def tile_index_case(B, hq, hkv, D, bs, lens, R=1, dtype="bf16", kv_dtype=None, seed=0):
    """q = 0, so every token a row sees weighs the same; V of token t in KV head h
    is one-hot at d = (t // 16 + h) % D. Output d of a row that sees Lr tokens is
    then (its tokens whose 16-token tile maps to d) / Lr exactly, and a tile read
    twice or not at all moves one output by 16 / Lr (6% of it at 32K tokens)."""
    case = pi.make_case(B, hq, hkv, D, bs, lens, dtype=dtype, seed=seed, device="cuda",
                        kv_dtype=kv_dtype, v_scale=1.0)
    if R > 1:
        case.q = torch.zeros((B, R, hq, D), dtype=case.q.dtype, device="cuda")
    else:
        case.q.zero_()
    fp8 = kv_dtype == "fp8"
    v = case.v_cache.view(torch.uint8) if fp8 else case.v_cache
    v.zero_()
    one = 0x38 if fp8 else 1.0  # E4M3 code of 1.0
    for b, L in enumerate(lens):
        t = torch.arange(L, device="cuda")
        phys = case.block_tables[b, t // bs].long()
        for h in range(hkv):
            v[phys, t % bs, h, (t // 16 + h) % D] = one
    return case


def tile_index_expected(lens, R, hq, hkv, D, window=0):
    B, G = len(lens), hq // hkv
    e = np.zeros((B, R, hq, D))
    for b, L in enumerate(lens):
        for i in range(R):
            Lr = L - R + i + 1
            if Lr <= 0:
                continue
            t = np.arange(max(0, Lr - window) if window else 0, Lr)
            Lr = len(t)
            for h in range(hq):
                e[b, i, h] = np.bincount((t // 16 + h // G) % D, minlength=D) / Lr
    return e if R > 1 else e[:, 0]


@pytest.mark.parametrize("B,hq,hkv,D,bs,lens,R,dtype,kv,splits,window", [
    (1, 8, 8, 128, 16, [32768], 1, "bf16", None, 0, 0),
    (1, 8, 8, 128, 16, [32763], 1, "f16", None, 0, 0),        # ragged last tile
    (1, 24, 4, 256, 784, [32768], 1, "bf16", None, 0, 0),
    (2, 16, 8, 128, 16, [32768, 20000], 1, "f16", None, 0, 0),  # shorter second sequence
    (1, 8, 8, 128, 16, [65536], 1, "bf16", "fp8", 0, 0),
    (1, 32, 8, 128, 16, [32768], 4, "bf16", None, 0, 0),      # four causal query rows
    (1, 8, 8, 128, 16, [32768], 1, "bf16", None, 2, 0),       # two long splits
    (1, 24, 4, 256, 784, [9000], 1, "bf16", None, 5, 0),
    (2, 8, 8, 128, 16, [32768, 30001], 1, "bf16", None, 0, 30000),  # sliding window
])
def test_shared_tiles_count_every_token_once(cuda_lib, B, hq, hkv, D, bs, lens, R, dtype, kv,
                                             splits, window):
    case = tile_index_case(B, hq, hkv, D, bs, lens, R=R, dtype=dtype, kv_dtype=kv)
    e = tile_index_expected(lens, R, hq, hkv, D, window=window)
    for det in (False, True):
        y = to_np(run(cuda_lib, case, splits=splits, deterministic=det, window=window))
        err = np.abs(y - e).max() / np.abs(e).max()
        assert err <= 1e-2, f"deterministic={det}: error {err:.2e} (a tile is 16 / L)"
    no_device_errors(cuda_lib)


# ------------------------------------------------------------------ invariances
def test_block_permutation_invariance(cuda_lib):
    case = pi.make_case(3, 32, 8, 128, 16, [3001, 17, 4096], seed=11, poison="kv_nan")
    y1 = run(cuda_lib, case, deterministic=True)
    y2 = run(cuda_lib, pi.repage(case, seed=12), deterministic=True)
    assert torch.equal(y1, y2), "the block table layout must not change a bit"
    case = pi.make_case(1, 24, 4, 256, 784, [6000], seed=13)
    assert torch.equal(run(cuda_lib, case, deterministic=True),
                       run(cuda_lib, pi.repage(case, seed=14), deterministic=True))
    case = pi.make_case(1, 8, 8, 128, 16, [32768], seed=16, device="cuda")  # shared tiles
    assert rel_diff(run(cuda_lib, case), run(cuda_lib, pi.repage(case, seed=17))) <= ORDER_TOL


def test_equal_scores_give_mean_of_v(cuda_lib):
    case = pi.make_case(1, 16, 8, 128, 16, [777], seed=15).to("cuda")
    case.q.zero_()
    y = to_np(run(cuda_lib, case))
    G = 2
    for h in range(16):
        mean = pi.to_f64_numpy(case.V[0][:, h // G, :]).mean(axis=0)
        assert np.abs(y[0, h] - mean).max() <= 1e-2 * np.abs(mean).max()


def test_one_hot_score_selects_row(cuda_lib):
    # K[t0] = c * q / |q|^2 per head with scale*c = 50, every other live K row zero:
    # softmax puts weight 1 - O(300 e^-50) on token t0, so out = V[t0].
    case = pi.make_case(1, 8, 8, 128, 16, [300], seed=16, dtype="f16")
    t0 = 123
    q = case.q[0].double()
    K = torch.zeros_like(case.K[0])
    for h in range(8):
        K[t0, h] = (50.0 / case.scale * q[h] / (q[h] @ q[h])).to(K.dtype)
    case.K[0].copy_(K)
    bt = case.block_tables[0].long()
    t = torch.arange(300)
    case.k_cache[bt[t // 16], t % 16] = case.K[0]
    y = to_np(run(cuda_lib, case))
    v = pi.to_f64_numpy(case.V[0][t0])
    assert np.abs(y[0] - v).max() <= 1e-2 * np.abs(v).max()


# ------------------------------------------------------------------ edge cases
def test_edge_lengths(cuda_lib):
    case = pi.make_case(6, 16, 8, 128, 16, [0, 1, 15, 16, 17, 0], seed=17, poison="kv_nan",
                        table_fill="oob")
    y = run(cuda_lib, case)
    assert torch.all(y[0] == 0) and torch.all(y[5] == 0)
    assert_parity(to_np(y), oracle_case(case), what="edge lengths")
    no_device_errors(cuda_lib)


def test_all_empty_batch(cuda_lib):
    case = pi.make_case(3, 8, 8, 128, 16, [0, 0, 0], seed=18)
    c = case.to("cuda")
    out = torch.full_like(c.q, float("nan"))
    cuda_lib.decode(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, c.scale,
                    out=out, max_seq_len=16)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_million_token_context(cuda_lib):
    # one KV head with 8 query heads over 2^20 - 3 tokens: hundreds of splits (more
    # than the merge keeps in registers), a shared tail, a ragged last tile
    L = (1 << 20) - 3
    case = pi.make_case(1, 8, 1, 128, 16, [L], seed=23, poison="kv_nan", device="cuda")
    S, P = cuda_lib.plan(1, 8, 1, 128, 16, L)
    assert S > 64
    y = run(cuda_lib, case)
    assert torch.isfinite(y).all()
    check_sampled(cuda_lib, case, y, [(0, 0)], "1M tokens")
    no_device_errors(cuda_lib)


def test_large_batch_of_short_sequences(cuda_lib):
    # 1024 sequences x 8 KV heads: more (sequence, KV head) pairs than the shared-tile
    # counters cover, lengths 0..200 including empty ones
    rng = np.random.default_rng(24)
    lens = [int(x) for x in rng.integers(0, 201, size=1024)]
    case = pi.make_case(1024, 16, 8, 128, 16, lens, seed=24, poison="v_nan", device="cuda")
    y = run(cuda_lib, case)
    assert torch.isfinite(y).all()
    pairs = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, 1024, 16), rng.integers(0, 8, 16))}
                   | {(int(np.argmax(lens)), 7)})
    check_sampled(cuda_lib, case, y, pairs, "large batch")
    for b in np.nonzero(np.array(lens) == 0)[0][:4]:
        assert torch.all(y[int(b)] == 0)
    no_device_errors(cuda_lib)


def test_block_size_one(cuda_lib):
    # every token in its own block: one table entry per token
    case = pi.make_case(2, 16, 4, 128, 1, [3001, 77], seed=25, poison="kv_nan")
    assert_parity(to_np(run(cuda_lib, case)), oracle_case(case), what="block size 1")
    case = pi.make_case(1, 24, 4, 256, 1, [1234], seed=26)
    assert_parity(to_np(run(cuda_lib, case)), oracle_case(case), what="block size 1, D 256")
    no_device_errors(cuda_lib)


@pytest.mark.parametrize("hq,hkv,D,bs,dtype", [
    (5, 1, 128, 16, "bf16"), (7, 1, 256, 16, "f16"), (16, 1, 128, 32, "bf16"),
    (12, 1, 256, 784, "bf16"), (32, 2, 128, 16, "f16"), (3, 3, 256, 48, "bf16"),
    (64, 64, 128, 16, "bf16"),
])
def test_other_shapes(cuda_lib, hq, hkv, D, bs, dtype):
    case = pi.make_case(2, hq, hkv, D, bs, [999, 2500], dtype=dtype, seed=19)
    assert_parity(to_np(run(cuda_lib, case)), oracle_case(case),
                  what=f"{hq}/{hkv} D={D} bs={bs} {dtype}")


def test_determinism(cuda_lib):
    case = pi.make_case(4, 24, 8, 128, 16, [5000, 300, 2048, 7777], seed=20).to("cuda")
    a = run(cuda_lib, case, deterministic=True)
    b = run(cuda_lib, case, deterministic=True)
    assert torch.equal(a, b)
    # long contexts at batch 1 share tiles: bitwise only in deterministic mode
    case = pi.make_case(1, 24, 4, 256, 784, [32768], seed=20, device="cuda")
    outs = [run(cuda_lib, case, deterministic=True) for _ in range(3)]
    assert all(torch.equal(o, outs[0]) for o in outs)
    for _ in range(3):
        assert rel_diff(run(cuda_lib, case), outs[0]) <= ORDER_TOL


def test_cuda_graph_replay(cuda_lib):
    case = pi.make_case(2, 32, 8, 128, 16, [4000, 2500], seed=21).to("cuda")
    ref = run(cuda_lib, case, deterministic=True)
    out = torch.empty_like(case.q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run_kw = dict(out=out, max_seq_len=case.max_seq_len, deterministic=True)
        cuda_lib.decode(case.q, case.k_cache, case.v_cache, case.block_tables, case.seq_lens,
                        case.scale, **run_kw)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            cuda_lib.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                            case.seq_lens, case.scale, **run_kw)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_graph_replays_rearm_the_tile_counters(cuda_lib):
    # a call whose splits share their tail, captured once and replayed: every replay
    # must find the counters at zero again (the merge grid rearms them)
    case = pi.make_case(1, 8, 8, 128, 16, [32768], seed=27, device="cuda")
    ref = run(cuda_lib, case, deterministic=True)
    check_sampled(cuda_lib, case, ref, [(0, 0), (0, 7)], "graph reference")
    out = torch.empty_like(case.q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kw = dict(out=out, max_seq_len=case.max_seq_len)
        cuda_lib.decode(case.q, case.k_cache, case.v_cache, case.block_tables, case.seq_lens,
                        case.scale, **kw)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                cuda_lib.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                case.seq_lens, case.scale, **kw)
    for _ in range(5):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert rel_diff(out, ref) <= ORDER_TOL
    no_device_errors(cuda_lib)


def test_two_streams_with_their_own_workspaces(cuda_lib):
    # sharing calls in flight on two streams at once, each with the binding's default
    # workspace of its stream (its own tile counters)
    cases = [pi.make_case(1, 8, 8, 128, 16, [32768 - 97 * i], seed=28 + i, device="cuda")
             for i in range(2)]
    refs = [run(cuda_lib, c, deterministic=True) for c in cases]
    streams = [torch.cuda.Stream() for _ in cases]
    outs = [torch.empty_like(c.q) for c in cases]
    torch.cuda.synchronize()
    for _ in range(4):
        for c, o, st in zip(cases, outs, streams):
            with torch.cuda.stream(st):
                cuda_lib.decode(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, c.scale,
                                out=o, max_seq_len=c.max_seq_len, stream=st)
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert rel_diff(o, r) <= ORDER_TOL
    for st in streams:
        ws = cuda_lib.default_workspace(cases[0].q.device, st)
        assert ws is not None and cuda_lib.read_device_errors(ws, stream=st) == 0


@pytest.mark.parametrize("shape", ["d128", "hybrid", "fp8", "window", "rows"])
def test_two_splits_merge_in_their_cluster(cuda_lib, shape):
    # Two splits run as one thread-block cluster and merge in distributed shared
    # memory, with no merge grid (both head_dims; fp8 caches with more than 16 columns
    # at head_dim 128 take the merge grid). Edge cases: an empty context, contexts where the
    # second split has no token (one of them, 1900, ends between the second split's
    # static start and the partition size, where a split past the sequence would
    # double-count tokens if it streamed its static share), a context shorter than a
    # tile, and a long one whose splits share their tail.
    lens = [0, 5, 33, 700, 1900, 4000]
    kw = dict(splits=2)
    if shape == "hybrid":
        case = pi.make_case(6, 24, 4, 256, 784, lens, seed=31, poison="kv_nan")
    elif shape == "fp8":
        case = pi.make_case(6, 32, 8, 128, 16, lens, seed=32, poison="kv_nan", kv_dtype="fp8")
    else:
        case = pi.make_case(6, 32, 16, 128, 16, lens, seed=33, poison="kv_nan")
    if shape == "window":
        kw["window"] = 1024
    if shape == "rows":
        case = rows_case(3, 6, 32, 16, 128, 16, lens, seed=34, poison="kv_nan")
        y = run(cuda_lib, case, **kw)
        ref = oracle_rows_case(case)
        assert_parity(to_np(y), ref, what="two splits, query rows")
    else:
        y = run(cuda_lib, case, **kw)
        ref = oracle_case(case, window=kw.get("window", 0))
        assert_parity(to_np(y), ref, what=f"two splits, {shape}")
    assert torch.isfinite(y).all()
    assert float(y[0].abs().max()) == 0.0  # the empty context
    # the same call through the merge grid (three splits) agrees
    kw3 = dict(kw, splits=3)
    y3 = run(cuda_lib, case, **kw3)
    assert rel_diff(y, y3) <= ORDER_TOL
    # and in deterministic mode repeated calls are bit-identical
    a = run(cuda_lib, case, deterministic=True, **kw)
    b = run(cuda_lib, case, deterministic=True, **kw)
    assert torch.equal(a, b)
    no_device_errors(cuda_lib)


@pytest.mark.parametrize("S", [3, 5, 8])
@pytest.mark.parametrize("shape", ["d128", "hybrid", "fp8"])
def test_splits_merge_in_their_cluster(cuda_lib, S, shape):
    # Three to eight splits of each (sequence, KV head) run as one thread-block
    # cluster when every cluster of the launch is resident at once: each split pushes
    # its state of every output item into the item's owner (distributed shared
    # memory) and the owners reduce, with no merge grid. Edge cases as for two splits:
    # an empty context, splits past the sequence, a context shorter than a tile.
    lens = [0, 5, 33, 700, 1900]
    if shape == "hybrid":  # 3 sequences x 4 KV heads: 12 clusters, all resident
        case = pi.make_case(3, 24, 4, 256, 784, [0, 33, 1900], seed=40 + S, poison="kv_nan")
    elif shape == "fp8":
        case = pi.make_case(5, 16, 2, 128, 16, lens, seed=41 + S, poison="kv_nan", kv_dtype="fp8")
    else:
        case = pi.make_case(5, 8, 2, 128, 16, lens, seed=42 + S, poison="kv_nan")
    c = case.to("cuda")
    assert cuda_lib.kernel_count(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens, c.scale,
                                 max_seq_len=c.max_seq_len, splits=S) == 1, "no merge grid"
    y = run(cuda_lib, c, splits=S)
    ref = oracle_case(case)
    assert_parity(to_np(y), ref, what=f"{S} splits in a cluster, {shape}")
    assert float(y[0].abs().max()) == 0.0  # the empty context
    # the merge grid (more splits than a cluster takes) agrees
    assert rel_diff(y, run(cuda_lib, c, splits=12)) <= ORDER_TOL
    a = run(cuda_lib, c, splits=S, deterministic=True)
    assert torch.equal(a, run(cuda_lib, c, splits=S, deterministic=True))
    no_device_errors(cuda_lib)


def test_kernel_count_follows_the_plan(cuda_lib):
    # one kernel for a single split or splits merging in their cluster, two with a
    # merge grid; the bench counts its launches through this call
    def count(B, hq, hkv, D, bs, L, **kw):
        c = pi.make_case(B, hq, hkv, D, bs, [L] * B, seed=7, device="cuda")
        return cuda_lib.kernel_count(c.q, c.k_cache, c.v_cache, c.block_tables, c.seq_lens,
                                     c.scale, max_seq_len=L, **kw)
    assert count(8, 32, 16, 128, 16, 8192) == 1          # one split per sequence
    assert count(8, 8, 8, 128, 16, 4096) == 1            # two splits, merged in clusters
    assert count(1, 24, 4, 256, 784, 500) == 1           # eight splits, four clusters
    assert count(1, 8, 8, 128, 16, 4096) == 2            # 19 splits: the merge grid
    assert count(8, 8, 8, 128, 16, 32768) == 2           # 7 splits of 64 pairs: not resident
    assert count(2, 8, 8, 128, 16, 4096, splits=1) == 1


def test_dependent_calls_back_to_back(cuda_lib):
    # Each call's query is the previous call's output, and a torch kernel rewrites a
    # live cache row (K and V) before every call. The calls follow each other with
    # programmatic dependent launch (a grid of single-split sequences lets the next
    # kernel launch after its main loop, a split grid its merge grid at once) and
    # share one workspace, so every call must still see the inputs of the kernels
    # before it complete. The chain runs as plain launches and as a captured graph;
    # both must equal, bit for bit, the chain with a device synchronisation between
    # all steps.
    case = pi.make_case(3, 16, 8, 128, 16, [4000, 700, 33], seed=29, device="cuda")
    splits = [1, 4, 1, 0, 2, 1, 7]
    blk = int(case.block_tables[1, 0])  # token 5 of sequence 1 lives in row 5 of this block
    g = torch.Generator(device="cpu").manual_seed(29)
    new_k = [torch.randn(8, 128, generator=g).to(case.k_cache.dtype).cuda() for _ in splits]
    new_v = [torch.randn(8, 128, generator=g).to(case.v_cache.dtype).cuda() for _ in splits]
    k0, v0, q0 = case.k_cache.clone(), case.v_cache.clone(), case.q.clone()
    k, v, q = case.k_cache, case.v_cache, case.q
    outs = [torch.empty_like(q) for _ in splits]
    max_len = case.max_seq_len  # read on the host before any capture

    def chain(sync):
        x = q
        for i, S in enumerate(splits):
            k[blk, 5].copy_(new_k[i])
            v[blk, 5].copy_(new_v[i])
            if sync:
                torch.cuda.synchronize()
            cuda_lib.decode(x, k, v, case.block_tables, case.seq_lens, case.scale, out=outs[i],
                            max_seq_len=max_len, splits=S, deterministic=True)
            if sync:
                torch.cuda.synchronize()
            x = outs[i]

    def restart():
        k.copy_(k0)
        v.copy_(v0)
        q.copy_(q0)
        for o in outs:
            o.fill_(float("nan"))

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        chain(sync=True)  # also sizes the stream's default workspace before the capture
        restart()
        chain(sync=True)
        ref = [o.clone() for o in outs]
        restart()
        chain(sync=False)
        s.synchronize()
        plain = [o.clone() for o in outs]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            chain(sync=False)
        restart()
        graph.replay()
        s.synchronize()
    for i, (r, a, b) in enumerate(zip(ref, plain, outs)):
        assert torch.isfinite(r).all(), f"call {i}"
        assert torch.equal(a, r), f"plain chain, call {i} (splits {splits[i]})"
        assert torch.equal(b, r), f"graph chain, call {i} (splits {splits[i]})"
    # the first call of the chain against the oracle on its inputs (the oracle reads the
    # contiguous K/V, so the rewritten row goes there too)
    case.K[1][5].copy_(new_k[0])
    case.V[1][5].copy_(new_v[0])
    assert_parity(to_np(ref[0]), oracle_case(case.to("cpu")), what="first call of the chain")
    ws = cuda_lib.default_workspace(q.device, s)
    assert ws is not None and cuda_lib.read_device_errors(ws, stream=s) == 0


# ------------------------------------------------------------------ sliding window
@pytest.mark.parametrize("W", [1, 16, 1000, 1024, 4096])
def test_sliding_window(cuda_lib, W):
    lens = [500, 1024, 1025, 4097, 9000]
    case = pi.make_case(5, 16, 8, 128, 16, lens, seed=50 + W, poison="kv_nan").to("cuda")
    y = run(cuda_lib, case, window=W)
    assert_parity(to_np(y), oracle_case(case, window=W), what=f"window {W}")
    no_device_errors(cuda_lib)


@pytest.mark.parametrize("L", [800, 5000, 32768])
def test_sliding_window_hybrid(cuda_lib, L):
    case = pi.make_case(1, 24, 4, 256, 784, [L], seed=L + 7, poison="v_nan")
    y = run(cuda_lib, case, window=1024)
    assert_parity(to_np(y), oracle_case(case, window=1024), what=f"hybrid window L={L}")


def test_window_never_attends_before_its_start(cuda_lib):
    # keys before the window get a huge score: attending to any of them would swamp
    # the output; the windowed result must match the oracle over the window alone
    W, L = 512, 3001
    case = pi.make_case(1, 8, 8, 128, 16, [L], seed=60)
    q = case.q[0].double()
    for h in range(8):
        case.K[0][: L - W, h] = (30.0 / case.scale * q[h] / (q[h] @ q[h])).to(case.K[0].dtype)
    bt = case.block_tables[0].long()
    t = torch.arange(L)
    case.k_cache[bt[t // 16], t % 16] = case.K[0]
    ref = oracle_case(case, window=W)
    y = run(cuda_lib, case, window=W)
    assert_parity(to_np(y), ref, what="window start")
    full = oracle_case(case)
    assert np.abs(full - ref).max() > 0.1 * np.abs(ref).max()   # the planted keys matter


@pytest.mark.parametrize("S", [1, 3, 7, 64])
def test_sliding_window_forced_splits(cuda_lib, S):
    case = pi.make_case(3, 32, 8, 128, 16, [2049, 700, 5000], seed=61).to("cuda")
    ref = oracle_case(case, window=1536)
    y = run(cuda_lib, case, splits=S, window=1536)
    assert_parity(to_np(y), ref, what=f"window splits={S}")


# ------------------------------------------------------------------ fp8 KV cache
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (8, 8)])
def test_fp8_cache_poison_matrix(cuda_lib, dtype, hq, hkv):
    lens = [1023, 4097]
    outs = {}
    for mode in pi.POISON_MODES:
        case = pi.make_case(2, hq, hkv, 128, 16, lens, dtype=dtype, seed=80, poison=mode,
                            kv_dtype="fp8")
        y = run(cuda_lib, case)
        if mode == "none":
            ref = oracle_case(case)
        assert_parity(to_np(y), ref, what=f"fp8 {mode} {dtype} {hq}/{hkv}")
        outs[mode] = run(cuda_lib, case, deterministic=True)
    for mode, y in outs.items():
        assert torch.equal(y, outs["none"]), f"fp8 output depends on the {mode} fill"
    no_device_errors(cuda_lib)


@pytest.mark.parametrize("L", [500, 5000, 32768])
def test_fp8_cache_hybrid(cuda_lib, L):
    case = pi.make_case(1, 24, 4, 256, 784, [L], seed=81, kv_dtype="fp8", poison="v_nan")
    assert_parity(to_np(run(cuda_lib, case)), oracle_case(case), what=f"fp8 hybrid L={L}")


def test_fp8_cache_scales_window_and_splits(cuda_lib):
    case = pi.make_case(3, 32, 16, 128, 16, [3000, 77, 6001], seed=82, kv_dtype="fp8",
                        k_scale=0.03, v_scale=0.05).to("cuda")
    assert_parity(to_np(run(cuda_lib, case)), oracle_case(case), what="fp8 scales")
    for S in (1, 5):
        assert_parity(to_np(run(cuda_lib, case, splits=S)), oracle_case(case),
                      what=f"fp8 splits={S}")
    assert_parity(to_np(run(cuda_lib, case, window=1024)), oracle_case(case, window=1024),
                  what="fp8 window")


def test_fp8_cache_mixed_batch_sampled(cuda_lib):
    lens = pi.uniform_seq_lens(64, 1024, 32768, seed=3)
    case = pi.make_case(64, 32, 8, 128, 16, lens, seed=83, pool_factor=1.1, poison="kv_nan",
                        device="cuda", kv_dtype="fp8")
    y = run(cuda_lib, case)
    assert torch.isfinite(y).all()
    rng = random.Random(3)
    pairs = sorted({(rng.randrange(64), rng.randrange(8)) for _ in range(8)})
    check_sampled(cuda_lib, case, y, pairs, "fp8 mixed batch")


# The fp8 kernels with more than one 8-column MMA tile. Queries with 17..32
# (row, head) columns at head_dim 128 take four column tiles (and cannot merge two
# splits in their cluster, so two splits go through the merge grid); 9..16 columns at
# head_dim 256 take two. Both query types, a straddling NaN tail, forced splits. The
# pages list an fp8 cache as untested ("vLLM's custom ROCm paged-attention kernel
# wins all sixty cells", §6).
FP8_WIDE = [
    # (R, hq, hkv, D, bs): columns = R * hq / hkv
    (8, 32, 8, 128, 16),     # 32 columns
    (2, 128, 8, 128, 16),    # 32 columns, G = 16
    (3, 48, 8, 128, 16),     # 18 columns (a partly used fourth tile)
    (1, 12, 1, 256, 784),    # 12 columns, head_dim 256
    (2, 24, 4, 256, 784),    # 12 columns, two rows of the hybrid layer
    (1, 64, 4, 256, 16),     # 16 columns
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("R,hq,hkv,D,bs", FP8_WIDE)
def test_fp8_cache_wide_column_tiles(cuda_lib, dtype, R, hq, hkv, D, bs):
    lens = [1023, 4097, 33] if D == 128 else [1567, 5000]

    def build(poison):
        kw = dict(dtype=dtype, poison=poison, kv_dtype="fp8")
        if R > 1:
            return rows_case(R, len(lens), hq, hkv, D, bs, lens, seed=110 + R + hq, **kw).to("cuda")
        return pi.make_case(len(lens), hq, hkv, D, bs, lens, seed=110 + hq, **kw).to("cuda")

    case = build("kv_nan")
    ref = oracle_rows_case(case) if R > 1 else oracle_case(case)
    for S in (0, 1, 2, 5):
        y = run(cuda_lib, case, splits=S)
        assert_parity(to_np(y), ref, what=f"fp8 {dtype} R={R} {hq}/{hkv} D={D} splits={S}")
    # the NaN fill of the unwritten tails and spare blocks must not change a bit
    assert torch.equal(run(cuda_lib, case, deterministic=True),
                       run(cuda_lib, build("none"), deterministic=True))
    no_device_errors(cuda_lib)


# The fp8 kernels move a column's running max only when a score exceeds it by more
# than 8 (log2 units), so weights reach 2^8 against a stale max. Keys along one
# direction with a growing coefficient make scores climb slowly across tiles (many
# tiles under the slack, then a rescale), jump (one tile far above), or fall (the max
# stays at the start); heads whose query points the other way see the mirror image.
def fp8_ramp_case(shape, hq, hkv, D, bs, lens, seed, R=1):
    kw = dict(seed=seed, kv_dtype="fp8", k_scale=1.0, poison="kv_nan")
    case = rows_case(R, len(lens), hq, hkv, D, bs, lens, **kw) if R > 1 else \
        pi.make_case(len(lens), hq, hkv, D, bs, lens, **kw)
    g = torch.Generator().manual_seed(seed)
    for b, L in enumerate(lens):
        t = torch.arange(L, dtype=torch.float32)
        if shape == "ramp":      # 0 .. 400 over the context
            a = 400.0 * t / max(L - 1, 1)
        elif shape == "jump":    # flat, then 300 higher from the middle on
            a = torch.where(t < L // 2, torch.zeros_like(t), torch.full_like(t, 300.0))
        else:                    # "fall": 400 down to 0
            a = 400.0 * (1.0 - t / max(L - 1, 1))
        k = torch.randn((L, hkv, D), generator=g)
        k[:, :, 0] = a[:, None]  # d = 0 carries the trend; e4m3 holds it coarsely
        codes = k.to(pi.FP8)     # k_scale = 1: stored values are the keys
        case.K[b] = codes
        bt = case.block_tables[b].long()
        phys = bt[t.long() // bs]
        case.k_cache[phys, t.long() % bs] = codes
    return case


@pytest.mark.parametrize("shape", ["ramp", "jump", "fall"])
@pytest.mark.parametrize("R,hq,hkv,D,bs", [(1, 32, 8, 128, 16), (1, 24, 4, 256, 784),
                                           (8, 32, 8, 128, 16)])
def test_fp8_rescale_slack(cuda_lib, shape, R, hq, hkv, D, bs):
    lens = [4097, 1500] if D == 128 else [5000, 1567]
    case = fp8_ramp_case(shape, hq, hkv, D, bs, lens, seed=120, R=R).to("cuda")
    ref = oracle_rows_case(case) if R > 1 else oracle_case(case)
    for S in (0, 1, 3):
        y = run(cuda_lib, case, splits=S)
        assert_parity(to_np(y), ref, what=f"fp8 {shape} R={R} {hq}/{hkv} D={D} splits={S}")
    no_device_errors(cuda_lib)


# ------------------------------------------------------------------ several query rows
def rows_case(R, *args, **kw):
    """A case whose q holds R query rows per sequence: [B, R, Hq, D]."""
    case = pi.make_case(*args, **kw)
    g = torch.Generator().manual_seed(1000 + R)
    B, Hq, D = case.q.shape
    case.q = torch.randn((B, R, Hq, D), generator=g).to(case.q.dtype).to(case.q.device)
    return case


@pytest.mark.parametrize("R,hq,hkv", [(2, 8, 8), (4, 16, 8), (4, 32, 8), (2, 64, 8),
                                      (8, 32, 8), (3, 24, 8)])
def test_query_rows(cuda_lib, R, hq, hkv):
    lens = [1, 3, 17, 1025, 4097]       # includes contexts shorter than R
    case = rows_case(R, 5, hq, hkv, 128, 16, lens, seed=90 + R, poison="kv_nan")
    y = run(cuda_lib, case)
    assert y.shape == case.q.shape
    assert_parity(to_np(y), oracle_rows_case(case), what=f"rows R={R} {hq}/{hkv}")
    no_device_errors(cuda_lib)


@pytest.mark.parametrize("S", [1, 3, 9])
def test_query_rows_splits_with_empty_columns(cuda_lib, S):
    # L = 33, 16-token splits: the last split holds tokens 32.. only, which row 0
    # (limit L - R + 1 = 30) cannot see
    case = rows_case(4, 2, 16, 8, 128, 16, [33, 100], seed=95).to("cuda")
    y = run(cuda_lib, case, splits=S)
    assert_parity(to_np(y), oracle_rows_case(case), what=f"rows splits={S}")


def test_query_rows_hybrid_and_fp8(cuda_lib):
    case = rows_case(2, 1, 24, 4, 256, 784, [5000], seed=96)
    assert_parity(to_np(run(cuda_lib, case)), oracle_rows_case(case), what="rows hybrid")
    case = rows_case(4, 3, 32, 8, 128, 16, [700, 4097, 9], seed=97, kv_dtype="fp8")
    assert_parity(to_np(run(cuda_lib, case)), oracle_rows_case(case), what="rows fp8")


def test_one_row_equals_single_query(cuda_lib):
    case = pi.make_case(3, 32, 8, 128, 16, [2000, 5, 3333], seed=98).to("cuda")
    a = run(cuda_lib, case, deterministic=True)
    q4 = case.q.unsqueeze(1).contiguous()
    b = cuda_lib.decode(q4, case.k_cache, case.v_cache, case.block_tables, case.seq_lens,
                        case.scale, max_seq_len=case.max_seq_len, deterministic=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b[:, 0])


# ------------------------------------------------------------------ device-side errors
def test_bad_block_index_is_reported_not_faulted(cuda_lib):
    case = pi.make_case(1, 8, 8, 128, 16, [100], seed=22).to("cuda")
    case.block_tables[0, 2] = case.num_blocks + 5     # a live token's block
    y = run(cuda_lib, case)
    assert torch.isfinite(y).all()
    assert cuda_lib.read_device_errors(cuda_lib.default_workspace()) == cuda_lib.PA_DEVERR_BLOCK_INDEX
    case.block_tables[0, 2] = -3
    run(cuda_lib, case)
    assert cuda_lib.read_device_errors(cuda_lib.default_workspace()) == cuda_lib.PA_DEVERR_BLOCK_INDEX


def test_seq_len_above_bound_is_reported(cuda_lib):
    case = pi.make_case(1, 8, 8, 128, 16, [100], seed=23).to("cuda")
    y = run(cuda_lib, case, max_seq_len=64)          # host bound smaller than the real length
    assert torch.isfinite(y).all()
    assert cuda_lib.read_device_errors(cuda_lib.default_workspace()) == cuda_lib.PA_DEVERR_SEQ_LEN


def test_host_errors_raise(cuda_lib):
    case = pi.make_case(1, 8, 8, 128, 16, [100], seed=24).to("cuda")
    with pytest.raises(cuda_lib.PAError):
        cuda_lib.decode(case.q, case.k_cache, case.v_cache, case.block_tables, case.seq_lens,
                        case.scale, max_seq_len=10 ** 6)
    with pytest.raises(ValueError):
        cuda_lib.decode(case.q.cpu(), case.k_cache, case.v_cache, case.block_tables,
                        case.seq_lens, case.scale)

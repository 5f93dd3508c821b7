"""The seeded input generator: paging scatter, fills, determinism (CPU only)."""
import numpy as np
import pytest
import torch

import pa_inputs as pi


def test_gather_back_inverts_scatter():
    case = pi.make_case(3, 8, 4, 16, 16, [37, 16, 1], seed=3)
    for b in range(case.B):
        k, v = pi.gather_back(case, b)
        assert torch.equal(k, case.K[b]) and torch.equal(v, case.V[b])


def test_gather_back_non_pow2_blocks():
    case = pi.make_case(2, 6, 1, 8, 784, [500, 1600], seed=4)
    for b in range(case.B):
        k, v = pi.gather_back(case, b)
        assert torch.equal(k, case.K[b]) and torch.equal(v, case.V[b])


def test_blocks_interleave_and_are_distinct():
    case = pi.make_case(4, 4, 4, 8, 16, [100, 64, 33, 200], seed=5)
    used = []
    for b in range(case.B):
        n = pi.blocks_for(int(case.seq_lens[b]), 16)
        used += case.block_tables[b, :n].tolist()
        assert all(x == -1 for x in case.block_tables[b, n:].tolist())
    assert len(used) == len(set(used)), "a physical block belongs to one sequence"
    assert all(0 <= x < case.num_blocks for x in used)


def test_first_config_structure():
    # 64-block cache, 32 blocks in a randomly permuted table, L=512, bs=16.
    case = pi.make_case(1, 8, 8, 128, 16, [512], seed=0, num_blocks=64)
    assert case.num_blocks == 64
    assert case.block_tables.shape == (1, 32)
    t = case.block_tables[0].tolist()
    assert sorted(t) != t, "the table is permuted"
    assert case.scale == np.float32(1 / np.sqrt(128))


@pytest.mark.parametrize("mode", pi.POISON_MODES)
def test_poison_lands_only_in_empty_slots(mode):
    bs = 16
    lens = [4090, 33]
    case = pi.make_case(2, 4, 2, 8, bs, lens, seed=6, poison=mode)
    kf = pi._fill_values(mode, "k", torch.bfloat16)
    vf = pi._fill_values(mode, "v", torch.bfloat16)
    occupied = torch.zeros(case.num_blocks, bs, dtype=torch.bool)
    for b, L in enumerate(lens):
        t = torch.arange(L)
        occupied[case.block_tables[b, t // bs].long(), t % bs] = True
        k, v = pi.gather_back(case, b)
        assert torch.equal(k, case.K[b]) and torch.equal(v, case.V[b])
    empty_k = case.k_cache[~occupied].float()
    empty_v = case.v_cache[~occupied].float()
    for arr, f in ((empty_k, kf), (empty_v, vf)):
        if f is None:
            assert torch.all(arr == 0)
        elif np.isnan(f):
            assert torch.all(torch.isnan(arr))
        else:
            assert torch.all(arr == torch.tensor(f, dtype=torch.bfloat16).float())
    # the unwritten tail of sequence 0's last block really is poisoned
    last = int(case.block_tables[0, pi.blocks_for(4090, bs) - 1])
    assert occupied[last].sum() == 16 - 6


def test_tail_slot_golden():
    from harness import read_golden
    for L, bs, n in read_golden("tail_slots.txt"):
        assert pi.unwritten_tail_slots(int(L), int(bs)) == int(n)


def test_determinism_and_seed_sensitivity():
    a = pi.make_case(2, 4, 2, 8, 16, [40, 7], seed=11)
    b = pi.make_case(2, 4, 2, 8, 16, [40, 7], seed=11)
    c = pi.make_case(2, 4, 2, 8, 16, [40, 7], seed=12)
    assert torch.equal(a.q, b.q) and torch.equal(a.k_cache, b.k_cache)
    assert torch.equal(a.block_tables, b.block_tables)
    assert not torch.equal(a.q, c.q)


def test_repage_keeps_tokens():
    a = pi.make_case(2, 4, 2, 8, 16, [70, 19], seed=13, poison="kv_nan")
    b = pi.repage(a, seed=99)
    assert not torch.equal(a.block_tables, b.block_tables)
    for i in range(2):
        k, v = pi.gather_back(b, i)
        assert torch.equal(k, a.K[i]) and torch.equal(v, a.V[i])


def test_empty_sequence_and_oob_table_fill():
    case = pi.make_case(3, 4, 4, 8, 16, [0, 5, 0], seed=14, table_fill="oob")
    assert case.block_tables[0].tolist() == [case.num_blocks + 7]
    assert case.K[0].shape == (0, 4, 8)


def test_uniform_seq_lens_range():
    lens = pi.uniform_seq_lens(64, 1024, 32768, seed=0)
    assert len(lens) == 64 and min(lens) >= 1024 and max(lens) <= 32768
    assert any(L % 16 for L in lens), "not block-aligned"


def test_fp8_case_roundtrip_and_fills():
    from harness import kv_f64
    case = pi.make_case(2, 8, 4, 16, 16, [37, 5], seed=70, kv_dtype="fp8", poison="kv_nan")
    assert case.k_cache.dtype == pi.FP8 and case.kv_fp8
    for b in range(2):
        k, v = pi.gather_back(case, b)
        assert torch.equal(k.view(torch.uint8), case.K[b].view(torch.uint8))
    kf = kv_f64(case, case.K[0], "k")
    # quantisation error of value / scale -> e4m3 is at most half an ulp (2^-4 relative)
    q = pi.make_case(2, 8, 4, 16, 16, [37, 5], seed=70)  # same draws, unquantised
    ref = q.K[0].double().numpy()
    assert np.all(np.abs(kf - ref) <= 2.0 ** -4 * np.abs(ref) + 2.0 ** -9 * case.k_scale)

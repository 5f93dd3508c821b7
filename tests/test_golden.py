"""Facts the pages print, checked against the arithmetic the build uses."""
from harness import kv_bytes, read_golden


def test_kv_bytes_per_token_formula():
    # bench.py and the roofline count KV bytes as L * Hkv * D * 2 * elem per layer.
    for layers, hkv, d, e, total in read_golden("kv_bytes_per_token.txt"):
        assert int(layers) * kv_bytes([1], int(hkv), int(d), int(e)) == int(total)
        assert int(total) == 64 * 1024


def test_block_size_784_is_not_pow2():
    for bs, a, b, is_pow2, d, g in read_golden("block_size_784.txt"):
        bs = int(bs)
        assert bs == int(a) * int(b)
        assert ((bs & (bs - 1)) == 0) == bool(int(is_pow2))
        assert bs % 16 == 0


def test_error_band_is_inside_the_bar():
    from harness import REL_LINF_TOL
    (lo, hi), = read_golden("error_band.txt")
    assert 0 < float(lo) < float(hi) < REL_LINF_TOL

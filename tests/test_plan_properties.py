"""Invariants of the launch plan over random arguments (CPU only; hypothesis)."""
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import paged_kv_attention_pa_gb300 as pa  # noqa: E402


@settings(max_examples=400, deadline=None)
@given(B=st.integers(1, 256), hkv=st.sampled_from([1, 2, 4, 8, 16, 32]),
       G=st.integers(1, 16), D=st.sampled_from([128, 256]),
       bs=st.sampled_from([1, 7, 16, 32, 784]), L=st.integers(1, 400_000),
       splits=st.sampled_from([0, 0, 0, 1, 2, 3, 7, 100, 5000]),
       fp8=st.booleans(), window=st.sampled_from([0, 0, 1, 100, 1024, 8192]),
       sms=st.sampled_from([1, 20, 132, 148, 152]), frac=st.floats(0.0, 1.0))
def test_plan_invariants(B, hkv, G, D, bs, L, splits, fp8, window, sms, frac):
    total = int(frac * B * L)
    S, P = pa.plan(B, G * hkv, hkv, D, bs, L, splits=splits, sm_count=sms, window=window,
                   kv_fp8=fp8, total_tokens=total)
    tile = 32 if (fp8 or D == 128) else 16
    span = min(L, window) if window else L       # tokens one sequence's splits cover
    assert P % tile == 0 and P >= tile            # whole warp tiles
    assert S * P >= span                          # the splits cover the longest context
    assert (S - 1) * P < span                     # and none of them is empty
    assert 1 <= S <= 1024                         # the merge's bound
    if splits == 0 and S > 1:
        assert P >= 64                            # automatic splits are not too short
    if splits > 0:
        assert S <= max(splits, -(-span // tile))  # forced: at most the request

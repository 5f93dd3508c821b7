"""Host-side helpers of bench.py (CPU only): the µs/call-vs-context fit and the
DRAM-traffic figure scaled from ncu captures."""
import bench


def test_linearity_fit_recovers_a_line():
    curve = [{"cell": f"hybrid L={L}", "us_per_call": 5.0 + 0.5 * L / 1024} for L in
             (500, 1024, 2048, 4096, 8192, 16384, 32768)]
    fit = bench.hybrid_linearity(curve)
    assert fit["range_tokens"] == [4096, 32768]      # only contexts >= 4K
    assert abs(fit["slope_us_per_1k_tokens"] - 0.5) < 1e-9
    assert abs(fit["intercept_us"] - 5.0) < 1e-9
    assert fit["r2"] == 1.0


def test_linearity_fit_needs_three_points_and_sees_curvature():
    assert bench.hybrid_linearity([{"cell": "hybrid L=4096", "us_per_call": 1.0}]) is None
    assert bench.hybrid_linearity([{"cell": "8/8 B=1 L=4096", "us_per_call": 1.0}] * 5) is None
    curve = [{"cell": f"hybrid L={L}", "us_per_call": (L / 1024) ** 2} for L in
             (4096, 8192, 16384, 32768)]
    assert bench.hybrid_linearity(curve)["r2"] < 0.99


def test_traffic_scaled_from_the_matching_capture(monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_SOURCES_SHA256", bench.kernel_sources_sha256())
    cap = bench.TRAFFIC_CAPTURES[(128, "bf16")]
    t, note = bench.traffic_per_call(cap["alg_bytes"], 128, "bf16")
    assert t == cap["dram_bytes"]
    assert "head_dim 128 bf16" in note
    assert bench.traffic_per_call(1e9, 64, "bf16")[0] is None   # no capture for the layout


def test_traffic_is_null_once_the_device_code_changes(monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_SOURCES_SHA256", "0" * 64)
    t, note = bench.traffic_per_call(1e9, 128, "bf16")
    assert t is None and "changed" in note


def test_source_fingerprint_ignores_comments_not_code():
    a = "int f(int x) {\n  return x + 1;  // one more\n}\n/* block\n comment */\n"
    b = "int f(int x) { return x + 1; }  // reworded comment\n"
    c = "int f(int x) { return x + 2; }\n"
    assert bench.code_tokens(a) == bench.code_tokens(b) == "int f(int x) { return x + 1; }"
    assert bench.code_tokens(c) != bench.code_tokens(a)


def test_captures_read_each_kv_byte_about_once():
    for (D, kv), cap in bench.TRAFFIC_CAPTURES.items():
        assert 1.0 <= cap["dram_bytes"] / cap["alg_bytes"] < 1.02, (D, kv)


def test_kernels_per_call_asks_the_library(monkeypatch):
    # the launch count is the library's own answer for the cell's tensors (which
    # depends on the device: splits merge in their clusters only when resident)
    import paged_kv_attention_pa_gb300 as pa
    seen = {}

    def fake_count(q, k, v, bt, sl, scale, max_seq_len=None, window=0, total_tokens=0):
        seen.update(q=q, k=k, max_seq_len=max_seq_len, window=window, total_tokens=total_tokens)
        return 2

    class Inst:
        q, k, v, bt, sl = "q", "k", "v", "bt", "sl"

    class Cell:
        insts = [Inst()]
        scale, max_len, window, total_tokens = 0.0625, 4096, 1024, 8192

    monkeypatch.setattr(pa, "kernel_count", fake_count)
    assert bench.kernels_per_call(pa, Cell()) == 2
    assert seen == dict(q="q", k="k", max_seq_len=4096, window=1024, total_tokens=8192)


def test_curve_summary_picks_the_batch1_and_mixed_cells():
    curve = [{"cell": "8/8 B=1 L=16384", "us_per_call": 14.0, "frac": 0.72},
             {"cell": "8/8 B=8 L=16384", "us_per_call": 90.0, "frac": 0.9},
             {"cell": "hybrid L=4096", "us_per_call": 6.0, "frac": 0.42,
              "ms_per_step_16_layers": 0.096},
             {"cell": "mixed B=64", "us_per_call": 700.0, "frac": 0.96}]
    s = bench.curve_summary(curve)
    assert s["batch1_8/8_frac"] == {"16384": 0.72}
    assert s["hybrid_us_per_call"] == {"4096": 6.0}
    assert s["hybrid_ms_per_step_16_layers"] == {"4096": 0.096}
    assert s["mixed_frac"] == 0.96 and s["mixed_us_per_call"] == 700.0
    assert "batch1_8/8_frac" in s and not any("B=8" in k for k in s)


def test_curve_summary_reports_fp8_against_bf16():
    curve = [{"cell": "hybrid L=32768", "us_per_call": 25.0, "frac": 0.8,
              "ms_per_step_16_layers": 0.4},
             {"cell": "fp8 hybrid L=32768", "us_per_call": 17.5, "frac": 0.57,
              "ms_per_step_16_layers": 0.28}]
    s = bench.curve_summary(curve)
    assert s["hybrid_us_per_call"] == {"32768": 25.0}     # the fp8 cell is not a bf16 one
    assert s["fp8_hybrid_us_per_call"] == {"32768": 17.5}
    assert s["fp8_over_bf16_hybrid_time"] == {"32768": 0.7}
    assert bench.hybrid_linearity(curve) is None            # fits only the bf16 cells

"""bench.py's roofline block on the CPU: the bound follows each workload's
algorithmic FLOP per byte against the ridge of the peaks, and the achieved
rate, the fraction and the units follow from it."""
import bench
import sdpa_inputs


def test_bound_follows_arithmetic_intensity():
    peak, hbm = 1890.0, 6770.0                      # TFLOP/s, GB/s: ridge ~279 FLOP/B
    bounds = {}
    for wid, w in sdpa_inputs.WORKLOADS.items():
        r = bench.roofline_of(w, w.flops(), 0.5, peak, hbm, "measured", None)
        bounds[wid] = r["bound"]
        assert abs(r["ridge_flop_per_byte"] - peak * 1e3 / hbm) < 1e-9
        assert abs(r["flop_per_byte"] - w.flops() / w.alg_bytes()) < 1e-9
        if r["bound"] == "hbm":
            assert r["unit"] == "GB/s" and r["peak"] == hbm
            assert abs(r["achieved"] - w.alg_bytes() / 0.5e-3 / 1e9) < 1e-6
        else:
            assert r["unit"] == "TFLOP/s" and r["peak"] == peak
            assert abs(r["achieved"] - w.flops() / 0.5e-3 / 1e12) < 1e-6
        assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    # 32 and 256 FLOP/B sit below the ridge; 910, 1024 and 4096 above it
    assert bounds == {1: "hbm", 2: "hbm", 3: "tensor", 4: "tensor", 5: "tensor"}


def test_without_a_bandwidth_peak_everything_is_tensor_bound():
    w = sdpa_inputs.WORKLOADS[2]
    assert bench.roofline_of(w, w.flops(), 1.0, 1890.0, 0.0, "fallback", None)["bound"] == "tensor"


def test_source_hash_ignores_comments_but_not_code():
    a = "int f() {  // one\n  return 1;\n}\n"
    b = "// a new header line\nint f() {  // two\n\n  return 1;\n}\n"
    c = "int f() {\n  return 2;\n}\n"
    assert bench.code_of(a) == bench.code_of(b)
    assert bench.code_of(a) != bench.code_of(c)

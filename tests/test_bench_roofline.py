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


def test_parity_block_passes_and_fails_on_the_tolerance():
    import numpy as np
    ref = np.linspace(-1.0, 1.0, 64).reshape(4, 16)
    ok = bench.parity_of(ref + 1e-4, ref, 4, "test")
    assert ok["pass"] and ok["rows"] == 4 and ok["max_abs"] < 2e-4
    bad = ref.copy()
    bad[2, 3] += 0.05                                   # one element past max-abs 2e-2
    assert not bench.parity_of(bad, ref, 4, "test")["pass"]
    nan = ref.copy()
    nan[0, 0] = np.nan
    assert not bench.parity_of(nan, ref, 4, "test")["pass"]
    assert not bench.parity_of(ref, ref, 4, "test", extra_ok=False, extra="dead rows")["pass"]


def test_oracle_sampler_rows_are_the_oracles_rows():
    """The CPU leg's sample (random (b, h, i) rows over every head) and the
    outputs it keeps for the parity check are the oracle's own rows."""
    import numpy as np
    import oracle
    w = sdpa_inputs.WORKLOADS[1]
    s = bench.OracleSampler(w)
    _, _, n = s.run(0.05, seed=3)
    assert s.last_rows.shape == (n, 3) and s.last_out.shape == (n, w.D)
    q, k, v, _ = sdpa_inputs.make(w)
    full = oracle.sdpa(q, k, v, is_causal=True)
    r = s.last_rows
    assert np.array_equal(full[r[:, 1], r[:, 2]], s.last_out)
    assert set(r[:, 1]) <= set(range(w.H)) and np.all(r[:, 0] == 0)


def test_l2_flush_follows_operand_size():
    import argparse
    a = argparse.Namespace(graph=False, flush_l2="auto")
    ws = sdpa_inputs.WORKLOADS
    assert [bench.flush_l2(a, ws[i]) for i in (1, 2, 3, 4, 5)] == [True, True, False, True, False]
    a.graph = True
    assert not bench.flush_l2(a, ws[2])

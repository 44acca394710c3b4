"""Host logic of bench.py that needs no GPU: the code-only source hash that keys the recorded
DRAM traffic, and the traffic lookup."""
import bench


def test_code_only_ignores_comments_and_blank_lines():
    a = "int f(int x) // doubles\n{\n    /* the\n       body */\n    return 2 * x;\n}\n"
    b = "int f(int x)\n{\n\n    return 2 * x;   \n}\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_only_sees_code_changes():
    a = "int f(int x) { return 2 * x; } // same comment\n"
    b = "int f(int x) { return 3 * x; } // same comment\n"
    assert bench._code_only(a) != bench._code_only(b)


def test_kernel_source_hash_is_stable_and_short():
    h = bench.kernel_source_hash()
    assert h == bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0


def test_recorded_traffic_is_an_int_or_none():
    for w in ("decode", "prefill", "no-such-workload"):
        v = bench.recorded_traffic(w)
        assert v is None or (isinstance(v, int) and v > 0)
    assert bench.recorded_traffic("no-such-workload") is None


def test_blas_baseline_computes_the_same_gemm_as_the_oracle():
    """The fp32 BLAS baseline dequantises on its own (numpy); on small problems its product
    agrees with the oracle's fp64 one within the GEMM tolerance, for u4b8 and u4, several
    group sizes."""
    import numpy as np
    import oracle
    import synth
    from helpers import within_tol
    orc = oracle.Oracle()
    for seed, (m, k, n, gs, wt) in enumerate([(3, 256, 256, 128, bench.U4B8),
                                              (5, 512, 256, 64, bench.U4),
                                              (2, 256, 512, -1, bench.U4B8)]):
        g = synth.group_count(k, gs)
        a = synth.activations(seed, m, k)
        qw = synth.qweight(seed, k, n)
        sc = synth.scales(seed, g, n)
        z = synth.zeros(seed, g, n) if wt == bench.U4 else None
        w = bench._dequant_fp32(qw, sc, z, gs, wt)
        got = a.astype(np.float64) @ w.astype(np.float64)
        ref = orc.gemm(a, qw, sc, z, None, gs, wt)
        ok, msg = within_tol(got, ref)
        assert ok, msg


def test_blas_sample_reports_the_tiny_workload():
    est, units, unit, text = bench.blas_sample("tiny", repeats=1)
    assert est > 0 and units > 0 and unit == "TFLOP/s" and "full M" in text

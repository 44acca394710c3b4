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
    for w in ("all:tcgen05", "all:column-slice", "no-such-workload"):
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
    est, text = bench.blas_sample("tiny", repeats=1)
    assert est > 0 and "full M" in text


def test_oracle_sample_and_cpu_line_on_the_tiny_workload():
    est, threads, text = bench.oracle_sample("tiny", 0.2)
    assert est > 0 and threads >= 1 and "two-point fit" in text
    peaks = bench.load_peaks()[0]
    line = bench.cpu_line("tiny", est, peaks)
    roof, flops, _ = bench.step_totals(bench.workload_specs("tiny"), peaks)
    assert abs(line["value"] - roof * 1e-6 / est) <= 1e-8 + 1e-6 * line["value"]
    assert line["tflops"] > 0


def test_roofline_per_gemm_takes_the_larger_bound():
    """max(bytes / HBM, flops / tensor peak) per GEMM: decode shapes are HBM-bound, M=4096
    prefill and the MoE pair tensor-bound, act-order M=1 HBM-bound."""
    peaks = {"hbm_gbs": 6784.8, "bf16_tflops": 1890.6}
    bound = {(s["config"], s.get("m")): bench.roofline_us(s, peaks)[1]
             for s in bench.workload_specs("all")}
    assert bound[("decode", 1)] == "hbm" and bound[("decode", 64)] == "hbm"
    assert bound[("prefill", 4096)] == "tensor" and bound[("actorder", 2048)] == "tensor"
    assert bound[("actorder", 1)] == "hbm" and bound[("actorder", 16)] == "hbm"
    s = bench.select_shape(bench.workload_specs("decode"), "1,4096,4096")[0]
    t, _ = bench.roofline_us(s, peaks)
    assert abs(t - bench.gemm_bytes(s) / 6784.8e3) < 1e-9


def test_all_workload_covers_every_configuration():
    specs = bench.workload_specs("all")
    assert {s["config"] for s in specs} == {"decode", "prefill", "actorder", "moe"}
    ms = sorted({s["m"] for s in specs if "m" in s})
    assert ms[0] == 1 and ms[-1] == 4096 and len(specs) == 12 + 6 + 3 + 2

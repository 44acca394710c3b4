"""Parity at the full workload sizes, in the launch configuration bench.py times.

Every GEMM is set up by bench.py's own DenseGemm / GroupedGemm (same inputs, flags and
dispatch as the timed run); the oracle then recomputes output rows and they must agree
elementwise within |c - ref| <= 1e-2 + 1e-2 |ref|.

Rows checked (dense): every row up to M = 256; above that the first and the last row of
every 16-row block -- every token tile of every kernel starts and ends on such a boundary
(tile heights are multiples of 16 rows) -- plus seeded random rows, at least 256 in all.
Grouped (MoE): every pair of the first and of the last active expert, and the first and
last pair of every other expert; the reference schedule is built by the oracle's own CSR
builder, not by the library's.

With W4A16_FULL_ORACLE=1 in the environment, `test_full_oracle_every_element` compares
every element of every configuration's output with the oracle (a few minutes of CPU time).
"""
import os

import numpy as np
import pytest

import bench
import oracle
import synth
from helpers import U4, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import weight_only_int4_03_gb300 as w4
    return w4


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def sample_rows(m: int, seed: int = 0):
    if m <= 256:
        return list(range(m))
    rows = set()
    for b in range(0, m, 16):
        rows.add(b)
        rows.add(min(b + 15, m - 1))
    rng = np.random.default_rng(seed + m)
    while len(rows) < 256:
        rows.add(int(rng.integers(0, m)))
    return sorted(rows)


def dense_inputs(spec, rows=None):
    """Oracle inputs of one dense GEMM of a workload (rows of A: all, or the given list)."""
    m, k, n, gs = spec["m"], spec["k"], spec["n"], spec["gs"]
    a = synth.activations(spec["seed"], m, k, sigma=spec["sigma"])
    if rows is not None:
        a = a[rows]
    qw = synth.qweight(spec["seed"], k, n)
    groups = synth.group_count(k, gs)
    scales = synth.scales(spec["seed"], groups, n)
    zeros = synth.zeros(spec["seed"], groups, n) if spec["wt"] == U4 else None
    g_idx = None
    if spec["act_order"]:
        g_idx = synth.act_order_gidx(synth.permutation(spec["seed"], k), gs)
    return np.ascontiguousarray(a), qw, scales, zeros, g_idx


def run_dense(w4, spec):
    import torch
    g = bench.DenseGemm(w4, spec, 1, torch.device("cuda"))
    g.run(0)
    torch.cuda.synchronize()
    assert w4.w4a16_status(g.ws) == 0
    return g


DENSE = [(wl, f"{s['m']},{s['k']},{s['n']}")
         for wl in ("decode", "prefill", "actorder", "fp8", "bf16") for s in bench.workload_specs(wl)]


def dense_reference(orc, spec, rows):
    """The oracle's rows `rows` (None: all) of one dense GEMM of bench.py's workloads, with the
    elementwise bar (atol = rtol) that applies: 1e-2, or 8e-2 for bf16 operands (R25)."""
    if spec["wt"] == bench.FE4M3:
        a = synth.activations(spec["seed"], spec["m"], spec["k"], sigma=spec["sigma"])
        if rows is not None:
            a = a[rows]
        qw = synth.fp8_weights(spec["seed"], spec["k"], spec["n"])
        s = synth.scales(spec["seed"], synth.group_count(spec["k"], spec["gs"]), spec["n"], 1e-4, 2e-4)
        return orc.gemm_fp8(np.ascontiguousarray(a), qw, s, spec["gs"]), 1e-2
    a, qw, scales, zeros, g_idx = dense_inputs(spec, rows)
    if spec.get("bf16"):
        # bench.py's bf16 operands: the same draws rounded to bfloat16
        bits = lambda x: synth.bf16_bits(np.asarray(x, dtype=np.float64))
        return orc.gemm_bf16(bits(a), qw, bits(scales), None if zeros is None else bits(zeros),
                             g_idx, spec["gs"], spec["wt"]), 8e-2
    return orc.gemm(a, qw, scales, zeros, g_idx, spec["gs"], spec["wt"]), 1e-2


def dense_output(g, spec, rows):
    c = g.c if rows is None else g.c[rows]
    if spec.get("bf16"):
        u = c.cpu().numpy().view(np.uint16).astype(np.uint32) << np.uint32(16)
        return u.view(np.float32).astype(np.float64)
    return c.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("workload,shape", DENSE)
def test_full_size_dense(w4, orc, workload, shape):
    spec = dict(bench.select_shape(bench.workload_specs(workload), shape)[0])
    g = run_dense(w4, spec)
    rows = sample_rows(spec["m"])
    ref, tol = dense_reference(orc, spec, rows)
    got = dense_output(g, spec, rows)
    ok, msg = within_tol(got, ref, tol, tol)
    assert ok, f"{workload} {shape} ({len(rows)} rows): {msg}"


def grouped_reference(orc, spec, g, pick_pairs):
    """The oracle's Y rows for the pairs `pick_pairs` (sorted), with the schedule rebuilt by
    the oracle from the same routes."""
    k, n, gs = spec["k"], spec["n"], spec["gs"]
    n_exp, n_tok, top_k = spec["n_exp"], spec["n_tok"], spec["top_k"]
    groups = synth.group_count(k, gs)
    sel = synth.routes(5000, n_tok, n_exp, top_k)
    ids, off, pairs, tok = orc.csr_from_token_routes(n_exp, n_tok, top_k, sel)
    if spec["pair_rows"]:
        tok = np.arange(n_tok * top_k, dtype=np.int32)
    a_all = synth.activations(spec["seed"], g.rows, k)
    scales = synth.scales(spec["seed"], n_exp * groups, n).reshape(n_exp, groups, n)
    want = set(pick_pairs)
    out = {}
    for i, e in enumerate(ids):
        seg = [int(p) for p in pairs[off[i]:off[i + 1]] if int(p) in want]
        if not seg:
            continue
        qw = synth.qweight(spec["seed"] * 100 + int(e), k, n)
        ref = orc.gemm(np.ascontiguousarray(a_all[tok[seg]]), qw, scales[e], None, None, gs,
                       spec["wt"])
        for r, p in enumerate(seg):
            out[p] = ref[r]
    return np.stack([out[p] for p in sorted(want)])


@pytest.mark.parametrize("index", [0, 1])
def test_full_size_grouped(w4, orc, index):
    """The MoE workload (8 experts, 512 tokens top-2): all pairs of the first and the last
    active expert, the first and last pair of every other expert."""
    import torch
    spec = dict(bench.workload_specs("moe")[index])
    g = bench.GroupedGemm(w4, spec, 1, torch.device("cuda"))
    g.run(0)
    torch.cuda.synchronize()
    assert w4.w4a16_status(g.ws) == 0
    sel = synth.routes(5000, spec["n_tok"], spec["n_exp"], spec["top_k"])
    ids, off, pairs, _ = orc.csr_from_token_routes(spec["n_exp"], spec["n_tok"], spec["top_k"], sel)
    pick = set()
    for i in range(len(ids)):
        seg = [int(p) for p in pairs[off[i]:off[i + 1]]]
        pick.update(seg if i in (0, len(ids) - 1) else (seg[0], seg[-1]))
    pick = sorted(pick)
    ref = grouped_reference(orc, spec, g, pick)
    got = g.c[pick].float().cpu().numpy().astype(np.float64)
    ok, msg = within_tol(got, ref)
    assert ok, f"moe[{index}] ({len(pick)} pairs): {msg}"


@pytest.mark.parametrize("index", [0, 1])
def test_full_size_moe_block_routing(w4, orc, index):
    """The MoE configuration through the block-routed (vLLM) interface, bench.py's moe_blocks
    workload: the same pairs as above against the oracle, the down projection's rows scaled by
    their top-k weights."""
    import torch
    spec = dict(bench.workload_specs("moe_blocks")[index])
    g = bench.GroupedGemm(w4, spec, 1, torch.device("cuda"))
    g.run(0)
    torch.cuda.synchronize()
    assert w4.w4a16_status(g.ws) == 0
    sel = synth.routes(5000, spec["n_tok"], spec["n_exp"], spec["top_k"])
    ids, off, pairs, _ = orc.csr_from_token_routes(spec["n_exp"], spec["n_tok"], spec["top_k"], sel)
    pick = set()
    for i in range(len(ids)):
        seg = [int(p) for p in pairs[off[i]:off[i + 1]]]
        pick.update(seg if i in (0, len(ids) - 1) else (seg[0], seg[-1]))
    pick = sorted(pick)
    ref = grouped_reference(orc, spec, g, pick)
    if g.topk_w is not None:
        ref = ref * g.topk_w.cpu().numpy().astype(np.float64)[pick][:, None]
    got = g.c[pick].float().cpu().numpy().astype(np.float64)
    ok, msg = within_tol(got, ref)
    assert ok, f"moe_blocks[{index}] ({len(pick)} pairs): {msg}"


FULL = os.environ.get("W4A16_FULL_ORACLE") == "1"


@pytest.mark.skipif(not FULL, reason="set W4A16_FULL_ORACLE=1 to compare every element")
@pytest.mark.parametrize("workload", ["tiny", "decode", "prefill", "actorder", "moe", "fp8", "bf16"])
def test_full_oracle_every_element(w4, orc, workload):
    import torch
    for spec in bench.workload_specs(workload):
        spec = dict(spec)
        if spec.get("grouped"):
            g = bench.GroupedGemm(w4, spec, 1, torch.device("cuda"))
            g.run(0)
            torch.cuda.synchronize()
            assert w4.w4a16_status(g.ws) == 0
            every = list(range(spec["n_tok"] * spec["top_k"]))
            ref = grouped_reference(orc, spec, g, every)
            got = g.c.float().cpu().numpy().astype(np.float64)
            what = f"moe k={spec['k']} n={spec['n']}"
        else:
            g = run_dense(w4, spec)
            ref, tol = dense_reference(orc, spec, None)
            got = dense_output(g, spec, None)
            what = f"{workload} m={spec['m']} k={spec['k']} n={spec['n']}"
        ok, msg = within_tol(got, ref, tol, tol) if not spec.get("grouped") else within_tol(got, ref)
        print(f"full oracle {what}: {got.size} elements, {msg}")
        assert ok, f"{what}: {msg}"
        del g
        torch.cuda.empty_cache()


def test_full_size_moe_swiglu_chain(w4, orc):
    """The chained MoE FFN of bench.py's moe_swiglu workload: gate_up with the SwiGLU epilogue
    writes H, the down projection reads H.  H is checked against the oracle's silu(gate) * up
    (the gated tolerance of test_gpu_glu), and the down output against the oracle's GEMM of the
    GPU's own H rows, on all pairs of the first and last expert and the first and last pair of
    every other.

    The down GEMM's input rows are not N(0, 1) like the configurations' A (H has an rms of about
    8 here).  The GEMM is linear in A and every rounding in it is relative to A's scale (the
    weights' fp16 products (q - z) s do not depend on A; the MMA products are exact), so the bar
    1e-2 + 1e-2 |ref| that holds for rows of rms 1 holds for A / r, i.e. 1e-2 r + 1e-2 |ref|
    for a row of rms r: that is the bar used here, with r = max(1, rms of the H row)."""
    import torch
    from test_gpu_glu import glu_check
    specs = [dict(s) for s in bench.workload_specs("moe_swiglu")]
    g0 = bench.GroupedGemm(w4, specs[0], 1, torch.device("cuda"))
    g1 = bench.GroupedGemm(w4, specs[1], 1, torch.device("cuda"))
    g1.a = g0.c
    g0.run(0)
    g1.run(0)
    torch.cuda.synchronize()
    assert w4.w4a16_status(g0.ws) == 0 and w4.w4a16_status(g1.ws) == 0
    s0 = specs[0]
    k, n2, gs, n_exp = s0["k"], s0["n"], s0["gs"], s0["n_exp"]
    i = n2 // 2
    groups = synth.group_count(k, gs)
    sel = synth.routes(5000, s0["n_tok"], n_exp, s0["top_k"])
    ids, off, pairs, tok = orc.csr_from_token_routes(n_exp, s0["n_tok"], s0["top_k"], sel)
    a_all = synth.activations(s0["seed"], s0["n_tok"], k)
    scales = synth.scales(s0["seed"], n_exp * groups, n2).reshape(n_exp, groups, n2)
    h_gpu = g0.c.float().cpu().numpy().astype(np.float64)
    picked = []
    for j, e in enumerate(ids):
        seg = [int(p) for p in pairs[off[j]:off[j + 1]]]
        if j not in (0, len(ids) - 1):
            seg = [seg[0], seg[-1]]
        picked += seg
        qw = synth.qweight(s0["seed"] * 100 + int(e), k, n2)
        rows = np.ascontiguousarray(a_all[tok[seg]])
        gate = orc.gemm(rows, np.ascontiguousarray(qw[:, :i]), np.ascontiguousarray(scales[e][:, :i]),
                        None, None, gs, s0["wt"])
        up = orc.gemm(rows, np.ascontiguousarray(qw[:, i:]), np.ascontiguousarray(scales[e][:, i:]),
                      None, None, gs, s0["wt"])
        glu_check(orc, h_gpu[seg], gate, up, 1)
    # down: y[p] = H[p] x dequant(B_down of p's expert), with the GPU's H as the input.
    s1 = specs[1]
    k1, n1 = s1["k"], s1["n"]
    groups1 = synth.group_count(k1, gs)
    scales1 = synth.scales(s1["seed"], n_exp * groups1, n1).reshape(n_exp, groups1, n1)
    h16 = g0.c.cpu().numpy()
    y = g1.c.float().cpu().numpy().astype(np.float64)
    for j, e in enumerate(ids):
        seg = [p for p in picked if p in set(int(x) for x in pairs[off[j]:off[j + 1]])]
        qw1 = synth.qweight(s1["seed"] * 100 + int(e), k1, n1)
        rows = np.ascontiguousarray(h16[seg])
        ref = orc.gemm(rows, qw1, scales1[e], None, None, gs, s1["wt"])
        r = np.maximum(1.0, np.sqrt(np.mean(rows.astype(np.float64) ** 2, axis=1)))[:, None]
        err = np.abs(y[seg] - ref)
        bound = 1e-2 * r + 1e-2 * np.abs(ref)
        assert np.all(np.isfinite(y[seg]))
        assert np.all(err <= bound), (f"down, expert {e}: {int((err > bound).sum())} outside, "
                                      f"max err/bound {float((err / bound).max()):.3f}")
        print(f"down expert {e}: max err {err.max():.3e}, max err/bound {(err / bound).max():.3f}, "
              f"row rms {float(r.min()):.2f}..{float(r.max()):.2f}")

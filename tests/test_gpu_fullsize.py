"""Parity at the full workload sizes, in the launch configuration bench.py times.

Every GEMM is set up by bench.py's own DenseGemm / GroupedGemm (same inputs, flags and
dispatch as the timed run); the oracle then recomputes sampled output rows one by one --
the first and last row, a middle row and the rows on each side of a token-tile boundary --
and they must agree elementwise within |c - ref| <= 1e-2 + 1e-2 |ref|.
"""
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


def sample_rows(m: int):
    rows = {0, m - 1, m // 2}
    for edge in (8, 16, 32, 64, 192, 208, 224, 256):   # token-tile heights of the two kernels
        if edge < m:
            rows.update((edge - 1, edge))
    return sorted(r for r in rows if 0 <= r < m)


DENSE = [
    ("decode", "1,4096,4096"), ("decode", "16,4096,4096"), ("decode", "32,4096,4096"),
    ("decode", "8,4096,12288"), ("decode", "32,4096,12288"), ("decode", "64,4096,12288"), ("prefill", "256,4096,11008"), ("prefill", "4096,4096,11008"),
    ("prefill", "4096,11008,4096"), ("actorder", "1,8192,28672"), ("actorder", "2048,8192,28672"),
]


@pytest.mark.parametrize("workload,shape", DENSE)
def test_full_size_dense(w4, orc, workload, shape):
    import torch
    spec = dict(bench.select_shape(bench.workload_specs(workload), shape)[0])
    g = bench.DenseGemm(w4, spec, 1, torch.device("cuda"))
    g.run(0)
    torch.cuda.synchronize()
    assert w4.w4a16_status(g.ws) == 0
    m, k, n, gs = spec["m"], spec["k"], spec["n"], spec["gs"]
    rows = sample_rows(m)
    a = synth.activations(spec["seed"], m, k, sigma=spec["sigma"])[rows]
    qw = synth.qweight(spec["seed"], k, n)
    groups = synth.group_count(k, gs)
    scales = synth.scales(spec["seed"], groups, n)
    zeros = synth.zeros(spec["seed"], groups, n) if spec["wt"] == U4 else None
    g_idx = None
    if spec["act_order"]:
        g_idx = synth.act_order_gidx(synth.permutation(spec["seed"], k), gs)
    ref = orc.gemm(np.ascontiguousarray(a), qw, scales, zeros, g_idx, gs, spec["wt"])
    got = g.c[rows].float().cpu().numpy().astype(np.float64)
    ok, msg = within_tol(got, ref)
    assert ok, f"{workload} {shape} rows {rows}: {msg}"


@pytest.mark.parametrize("index", [0, 1])
def test_full_size_grouped(w4, orc, index):
    """The MoE workload (8 experts, 512 tokens top-2): the first and last pair of every expert
    segment, each against the oracle's dense product with that expert's weights."""
    import torch
    spec = dict(bench.workload_specs("moe")[index])
    g = bench.GroupedGemm(w4, spec, 1, torch.device("cuda"))
    g.run(0)
    torch.cuda.synchronize()
    assert w4.w4a16_status(g.ws) == 0
    k, n, gs = spec["k"], spec["n"], spec["gs"]
    groups = synth.group_count(k, gs)
    ids, off, pairs, tok = (x.cpu().numpy() for x in g.csr)
    a_all = synth.activations(spec["seed"], g.rows, k)
    scales = synth.scales(spec["seed"], spec["n_exp"] * groups, n).reshape(spec["n_exp"], groups, n)
    got_all = g.c.float().cpu().numpy().astype(np.float64)
    for i, e in enumerate(ids):
        seg = pairs[off[i]:off[i + 1]]
        pick = sorted({int(seg[0]), int(seg[-1])})
        a = a_all[tok[pick]]
        qw = synth.qweight(spec["seed"] * 100 + int(e), k, n)
        ref = orc.gemm(np.ascontiguousarray(a), qw, scales[e], None, None, gs, spec["wt"])
        ok, msg = within_tol(got_all[pick], ref)
        assert ok, f"moe[{index}] expert {e} pairs {pick}: {msg}"

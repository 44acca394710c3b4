"""Back-to-back calls of different GEMMs on one stream, with no synchronisation between them.

Consecutive kernels overlap (programmatic dependent launch: a kernel's set-up, and with static
weights its first weight copies, run while the previous kernel drains), and every pipeline
barrier of the tcgen05 kernel is exercised through many phases.  Each workload's GEMMs run in
bench.py's order for a number of steps; every call must leave its workspace status clear and its
output equal, bit for bit, to the same call made alone (the kernels are deterministic).
"""
import numpy as np
import pytest

import bench

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import weight_only_int4_03_gb300 as w4
    return w4


@pytest.mark.parametrize("workload", ["fp8", "moe", "prefill", "bf16"])
def test_back_to_back_steps_match_single_calls(w4, workload):
    import torch
    dev = torch.device("cuda")
    gemms = []
    for s in bench.workload_specs(workload):
        s = dict(s)
        gemms.append(bench.GroupedGemm(w4, s, 1, dev) if s.get("grouped") else bench.DenseGemm(w4, s, 1, dev))
    alone = []
    for g in gemms:
        g.run(0)
        torch.cuda.synchronize()
        assert w4.w4a16_status(g.ws) == 0
        alone.append(g.c.clone())
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for step in range(12):
            for g in gemms:
                g.run(0)
    torch.cuda.synchronize()
    for g, ref in zip(gemms, alone):
        assert w4.w4a16_status(g.ws) == 0
        assert torch.equal(g.c.view(torch.int16), ref.view(torch.int16))

"""w4a16_gemm_noalloc, the entry point for callers that cannot allocate device memory (code
inside a host callback or an allocator hook, under a sealed memory pool, or in a plug-in whose
host gives it no workspace): its scratch is a fixed array inside the library.  Checked here,
through the C ABI and on two calls in a row, against the CPU oracle and against w4a16_gemm
with a caller-owned workspace, both within the GEMM tolerance.

Kept in a file of its own, collected after every other test file.
"""
import numpy as np
import pytest

import oracle
from helpers import FLAG_FORCE_TC, U4, DeviceProblem, make_problem, oracle_ref, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import weight_only_int4_03_gb300 as w4
    return w4


CASES = [
    dict(m=1, k=1024, n=768),
    dict(m=8, k=2048, n=512, act_order=True, group_size=64),
    dict(m=16, k=4096, n=4096),
    dict(m=33, k=768, n=512, weight_type=U4, sigma=0.5),
    dict(m=64, k=1024, n=1024),
    dict(m=96, k=512, n=256, flags=FLAG_FORCE_TC),
    dict(m=200, k=1024, n=512),
    dict(m=240, k=4096, n=512),               # one 240-row tile in w4a16_gemm, two of 192 here
    dict(m=600, k=1024, n=512),
    dict(m=1024, k=1024, n=768, group_size=64),  # 208-row tiles in w4a16_gemm, 192 here
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"m{c['m']}k{c['k']}n{c['n']}")
def test_noalloc_matches_workspace_entry_point(w4, case):
    import torch
    case = dict(case)
    extra = case.pop("flags", 0)
    m, k, n = case.pop("m"), case.pop("k"), case.pop("n")
    pb = make_problem(4000 + m, m, k, n, **case)
    exact = oracle_ref(oracle.Oracle(), pb)
    dp = DeviceProblem(w4, pb, flags_extra=extra)
    dp.run()
    ref = dp.result()
    assert dp.status() == 0

    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        c = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
        w4.w4a16_gemm_noalloc(dp.a, dp.b, c, dp.scales, dp.zeros, dp.g_idx, dp.perm, m, n, k,
                              pb.group_size, pb.weight_type, dp.flags, status_out=status)
        torch.cuda.synchronize()
        got = c.float().cpu().numpy().astype(np.float64)
        ok, msg = within_tol(got, exact)
        assert ok, f"vs oracle: {msg}"
        ok, msg = within_tol(got, ref)
        assert ok, f"vs w4a16_gemm: {msg}"
        assert int(status.item()) == 0


def test_noalloc_rejects_calls_beyond_its_scratch(w4):
    """An act-order call whose copy of A (M*K*2 = 8 MiB here) does not fit beside the partial
    slots is refused before anything launches."""
    import torch
    m, k, n, gs = 1024, 4096, 4096, 128
    flags = w4.W4A16_FLAG_ACT_ORDER | w4.W4A16_FLAG_IS_K_FULL
    assert w4.w4a16_workspace_size(m, n, k, gs, flags) > w4.W4A16_NOALLOC_SCRATCH_BYTES
    a = torch.zeros((m, k), dtype=torch.float16, device="cuda")
    b = torch.zeros(k * n // 8, dtype=torch.int32, device="cuda")
    s = torch.ones((k // gs, n), dtype=torch.float16, device="cuda")
    g_idx = (torch.arange(k, dtype=torch.int32, device="cuda") // gs).to(torch.int32)
    perm = torch.arange(k, dtype=torch.int32, device="cuda")
    c = torch.full((m, n), 5.0, dtype=torch.float16, device="cuda")
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemm_noalloc(a, b, c, s, None, g_idx, perm, m, n, k, gs, w4.W4A16_TYPE_U4B8,
                              flags)
    assert e.value.stage == 2 and e.value.detail == w4.W4A16_ARG_SCRATCH
    torch.cuda.synchronize()
    assert float(c.float().min()) == 5.0 and float(c.float().max()) == 5.0

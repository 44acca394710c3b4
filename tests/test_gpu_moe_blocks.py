"""Block-routed MoE (the vLLM Marlin-MoE routing interface) against the oracle, through the C ABI.

The routing comes from the library's host builder (checked against the oracle's on the CPU);
the reference output is the oracle's block-routed GEMM on the same routing.  Every row the
routing names must match within |c - ref| <= 1e-2 + 1e-2 |ref|; every other row of c keeps its
initial NaN (the call writes nothing there).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import FLAG_HAS_ZP, FLAG_IS_K_FULL, U4, U4B8, torch_dev, within_tol

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


def make_experts(seed, n_exp, k, n, wt, gs=128):
    groups = k // gs
    qw = np.stack([synth.qweight(seed * 10 + e, k, n) for e in range(n_exp)])
    s = synth.scales(seed, n_exp * groups, n).reshape(n_exp, groups, n)
    z = synth.zeros(seed, n_exp * groups, n).reshape(n_exp, groups, n) if wt == U4 else None
    return qw, s, z


def run_blocks(w4, a, qw, s, z, sid, eid, padded, tw, bs, top_k, is_ep, n_exp, k, n, wt,
               max_padded=None, flags_extra=0, gs=128, ntpp_value=None):
    import torch
    m = a.shape[0]
    max_padded = max_padded or padded
    b = torch.empty(n_exp * k * n // 8, dtype=torch.int32, device="cuda")
    per = k * n // 8
    for e in range(n_exp):
        w4.w4_repack(torch_dev(qw[e]), None, b[e * per:(e + 1) * per], k, n)
    sid_full = np.full(max_padded, m * top_k, np.int32)
    sid_full[:padded] = sid
    eid_full = np.zeros(max(max_padded // bs, 1), np.int32)
    eid_full[:len(eid)] = eid
    ntpp = torch.tensor([padded if ntpp_value is None else ntpp_value], dtype=torch.int32, device="cuda")
    flags = FLAG_IS_K_FULL | (FLAG_HAS_ZP if z is not None else 0) | flags_extra
    glu = flags & (w4.W4A16_FLAG_SWIGLU | w4.W4A16_FLAG_GEGLU)
    n_out = n // 2 if glu else n
    ws = torch.zeros(w4.w4a16_moe_blocks_workspace_size(max_padded, bs, n_exp, n, k, gs, flags),
                     dtype=torch.uint8, device="cuda")
    c = torch.full((m * top_k, n_out), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a16_gemm_moe_blocks(torch_dev(a), b, c, torch_dev(s.reshape(-1, n)),
                             torch_dev(z.reshape(-1, n)) if z is not None else None,
                             torch_dev(sid_full), torch_dev(eid_full), ntpp,
                             torch_dev(tw) if tw is not None else None, max_padded, bs, top_k,
                             tw is not None, is_ep, n_exp, m, n, k, gs, wt, flags, ws)
    torch.cuda.synchronize()
    return c.float().cpu().numpy().astype(np.float64), w4.w4a16_status(ws)


def compare(got, ref):
    named = ~np.isnan(ref[:, 0])
    assert np.all(np.isnan(got[~named])), "a row no entry names was written"
    ok, msg = within_tol(got[named], ref[named])
    assert ok, msg
    return int(named.sum())


@pytest.mark.parametrize("m,top_k,n_exp,bs,wt,weighted,n,k", [
    (100, 2, 4, 16, U4B8, False, 512, 512),
    (60, 3, 8, 64, U4, True, 256, 1024),
    (33, 2, 6, 8, U4B8, True, 768, 256),
    (5, 1, 1, 16, U4B8, False, 256, 256),       # the page's shape: one block, batch prefix
    (700, 2, 8, 48, U4B8, False, 512, 512),     # several token tiles per expert
])
def test_moe_blocks_matches_oracle(w4, orc, m, top_k, n_exp, bs, wt, weighted, n, k):
    seed = 7000 + m
    ids = synth.routes(seed, m, n_exp, top_k) if n_exp > 1 else np.zeros(m * top_k, np.int32)
    a = synth.activations(seed, m, k, sigma=0.5 if wt == U4 else 1.0)
    qw, s, z = make_experts(seed, n_exp, k, n, wt)
    tw = (synth.scales(seed + 1, 1, m * top_k, lo=0.1, hi=1.0).astype(np.float32).ravel()
          if weighted else None)
    sid, eid, padded = w4.w4a16_moe_align_block_size(ids, m, top_k, n_exp, bs)
    got, status = run_blocks(w4, a, qw, s, z, sid, eid, padded, tw, bs, top_k, False, n_exp, k, n, wt,
                             max_padded=padded + 2 * bs)
    assert status == 0
    ref = orc.moe_blocks(a, qw.ravel(), s, z, sid, eid, padded, tw, bs, top_k, False, n_exp, k, n,
                         128, wt)
    assert compare(got, ref) == m * top_k


def test_moe_blocks_expert_parallel_skips_blocks(w4, orc):
    """is_ep: blocks whose expert id is -1 are dropped; their rows stay unwritten."""
    m, top_k, n_exp, bs, k, n = 80, 2, 6, 16, 512, 256
    ids = synth.routes(7100, m, n_exp, top_k)
    a = synth.activations(7100, m, k)
    qw, s, z = make_experts(7100, n_exp, k, n, U4B8)
    sid, eid, padded = w4.w4a16_moe_align_block_size(ids, m, top_k, n_exp, bs)
    eid = eid.copy()
    eid[eid == 1] = -1
    eid[eid == 4] = -1
    got, status = run_blocks(w4, a, qw, s, z, sid, eid, padded, None, bs, top_k, True, n_exp, k, n, U4B8)
    assert status == 0
    ref = orc.moe_blocks(a, qw.ravel(), s, z, sid, eid, padded, None, bs, top_k, True, n_exp, k, n)
    named = compare(got, ref)
    assert 0 < named < m * top_k


@pytest.mark.parametrize("kind", [1, 2])
def test_moe_blocks_gated_and_weighted(w4, orc, kind):
    """The gated epilogue through the block routing (interleaved gate/up experts), with top-k
    weights: c[id] = act(gate) * up * w[id]."""
    import torch
    from test_gpu_glu import glu_check
    m, top_k, n_exp, bs, k, n2 = 64, 2, 4, 16, 512, 512
    i = n2 // 2
    ids = synth.routes(7200 + kind, m, n_exp, top_k)
    a = synth.activations(7200 + kind, m, k)
    qw, s, _ = make_experts(7200 + kind, n_exp, k, n2, U4B8)
    qw_i = np.stack([w4_interleave(w4, qw[e], n2) for e in range(n_exp)])
    s_i = np.stack([w4_interleave(w4, s[e], n2) for e in range(n_exp)])
    tw = (np.arange(m * top_k, dtype=np.float32) % 7 + 1) / 8
    sid, eid, padded = w4.w4a16_moe_align_block_size(ids, m, top_k, n_exp, bs)
    flag = w4.W4A16_FLAG_SWIGLU if kind == 1 else w4.W4A16_FLAG_GEGLU
    got, status = run_blocks(w4, a, qw_i, s_i, None, sid, eid, padded, tw, bs, top_k, False, n_exp,
                             k, n2, U4B8, flags_extra=flag)
    assert status == 0
    gate = orc.moe_blocks(a, np.ascontiguousarray(qw[:, :, :i]).ravel(), np.ascontiguousarray(s[:, :, :i]),
                          None, sid, eid, padded, None, bs, top_k, False, n_exp, k, i)
    up = orc.moe_blocks(a, np.ascontiguousarray(qw[:, :, i:]).ravel(), np.ascontiguousarray(s[:, :, i:]),
                        None, sid, eid, padded, tw, bs, top_k, False, n_exp, k, i)
    glu_check(orc, got, gate, up, kind)
    del torch


def w4_interleave(w4, x, n2):
    import torch
    src = torch_dev(x)
    dst = torch.empty_like(src)
    w4.w4_gate_up_interleave(src, dst, x.shape[0], n2)
    return dst.cpu().numpy()


def test_moe_blocks_bad_padded_length_reported(w4):
    """A padded length beyond the capacity (or not whole blocks) is reported and nothing is
    written."""
    m, top_k, n_exp, bs, k, n = 16, 2, 2, 16, 256, 256
    ids = synth.routes(7300, m, n_exp, top_k)
    a = synth.activations(7300, m, k)
    qw, s, z = make_experts(7300, n_exp, k, n, U4B8)
    sid, eid, padded = w4.w4a16_moe_align_block_size(ids, m, top_k, n_exp, bs)
    for bad in (padded + bs, padded - 3):
        got, status = run_blocks(w4, a, qw, s, z, sid, eid, padded, None, bs, top_k, False, n_exp,
                                 k, n, U4B8, ntpp_value=bad)
        assert status & w4.W4A16_DEV_SCHEDULE
        assert np.all(np.isnan(got))

"""Gated FFN epilogue (W4A16_FLAG_SWIGLU / _GEGLU) against the oracle, through the C ABI.

The gate and up projections of a planar [K, 2I] weight (gate columns first, then up) are
interleaved on the device by w4_gate_up_interleave (codes, scales, zeros), repacked, and run as
one GEMM whose epilogue writes H = act(A Wg) * (A Wu).  The oracle computes the two GEMMs on
the planar halves in fp64 and applies act(gate) * up.

Tolerance.  Each of gate and up meets the GEMM bar tau(x) = 1e-2 + 1e-2 |x| elementwise;
carried through h = act(g) u to first order, with |act'| <= 1.2 for both SiLU and the tanh
form of GELU, plus the fp16 rounding of h:
    |h - h_ref| <= 1e-2 + 1e-2 |h_ref| + 1.2 |u| tau(g) + |act(g)| tau(u) + 1.2 tau(g) tau(u)
with g, u, h the oracle's values.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import FLAG_FORCE_MMA, FLAG_IS_K_FULL, FLAG_HAS_ZP, U4, U4B8, torch_dev

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


def glu_check(orc, got, g, u, kind):
    h = orc.glu(g, u, kind)
    act = orc.glu(g, np.ones_like(u), kind)
    tau_g = 1e-2 + 1e-2 * np.abs(g)
    tau_u = 1e-2 + 1e-2 * np.abs(u)
    bound = 1e-2 + 1e-2 * np.abs(h) + 1.2 * np.abs(u) * tau_g + np.abs(act) * tau_u + 1.2 * tau_g * tau_u
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == h.shape
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - h)
    bad = err > bound
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{int(bad.sum())} of {bad.size} outside: first {idx} got {got[idx]} "
                             f"want {h[idx]} (g {g[idx]}, u {u[idx]}), max err {err.max():.3e}")
    return float(err.max())


def interleave_on_device(w4, planar, n2):
    import torch
    src = torch_dev(planar)
    dst = torch.empty_like(src)
    w4.w4_gate_up_interleave(src, dst, planar.shape[0], n2)
    return dst


@pytest.mark.parametrize("rows,n2,dtype", [(3, 64, np.int32), (5, 512, np.float16), (1, 32, np.int32)])
def test_interleave_is_the_block_permutation(w4, rows, n2, dtype):
    """Column 32b + r takes gate column 16b + r (r < 16) or up column 16b + r - 16, bit for bit."""
    rng = np.random.default_rng(rows * n2)
    x = rng.integers(-2**31, 2**31 - 1, size=(rows, n2), dtype=np.int64).astype(np.int32)
    if dtype == np.float16:
        x = (x & 0x7BFF).astype(np.uint16).view(np.float16)
    got = interleave_on_device(w4, x, n2).cpu().numpy()
    half = n2 // 2
    want = np.empty_like(x)
    for j in range(n2):
        b, r = divmod(j, 32)
        want[:, j] = x[:, 16 * b + r] if r < 16 else x[:, half + 16 * b + r - 16]
    assert np.array_equal(got.view(np.uint8), want.view(np.uint8))


def run_glu(w4, a, qw, s, z, k, n2, gs, wt, kind, extra=0):
    """One gated call on planar weights (interleaved and repacked on the device)."""
    import torch
    m = a.shape[0]
    qw_i = interleave_on_device(w4, qw, n2)
    s_i = interleave_on_device(w4, s, n2)
    z_i = interleave_on_device(w4, z, n2) if z is not None else None
    b = torch.empty(k * n2 // 8, dtype=torch.int32, device="cuda")
    w4.w4_repack(qw_i, None, b, k, n2)
    flags = FLAG_IS_K_FULL | (FLAG_HAS_ZP if z is not None else 0) | extra
    flags |= w4.W4A16_FLAG_SWIGLU if kind == 1 else w4.W4A16_FLAG_GEGLU
    ws = torch.zeros(w4.w4a16_workspace_size(m, n2, k, gs, flags), dtype=torch.uint8, device="cuda")
    h = torch.full((m, n2 // 2), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a16_gemm(torch_dev(a), b, h, s_i, z_i, None, None, ws, m, n2, k, gs, wt, flags)
    torch.cuda.synchronize()
    assert w4.w4a16_status(ws) == 0
    return h.float().cpu().numpy().astype(np.float64), (b, s_i, z_i, flags, ws)


@pytest.mark.parametrize("m,k,n2,wt,kind", [
    (1, 512, 512, U4B8, 1),       # split tiles (4 column tiles, many CTAs each)
    (40, 2048, 512, U4, 1),       # u4 zeros, split tiles
    (300, 512, 1024, U4B8, 1),    # two token tiles, split
    (4096, 256, 2048, U4B8, 1),   # 304 whole tiles: the tile epilogue
    (16, 1024, 768, U4B8, 2),     # GeGLU, split
    (1000, 256, 4096, U4, 2),     # GeGLU, u4, whole tiles
])
def test_gated_gemm_matches_oracle(w4, orc, m, k, n2, wt, kind):
    gs = 128
    seed = 6000 + m + n2
    groups = k // gs
    i = n2 // 2
    a = synth.activations(seed, m, k, sigma=0.5 if wt == U4 else 1.0)
    qw = synth.qweight(seed, k, n2)
    s = synth.scales(seed, groups, n2)
    z = synth.zeros(seed, groups, n2) if wt == U4 else None
    got, _ = run_glu(w4, a, qw, s, z, k, n2, gs, wt, kind)
    g = orc.gemm(a, np.ascontiguousarray(qw[:, :i]), np.ascontiguousarray(s[:, :i]),
                 None if z is None else np.ascontiguousarray(z[:, :i]), None, gs, wt)
    u = orc.gemm(a, np.ascontiguousarray(qw[:, i:]), np.ascontiguousarray(s[:, i:]),
                 None if z is None else np.ascontiguousarray(z[:, i:]), None, gs, wt)
    glu_check(orc, got, g, u, kind)


def test_gated_flags_rejected(w4):
    """Both activations at once, or the gated epilogue with a small-M kernel forced, are
    rejected before anything launches; so is an output narrower than I."""
    import torch
    k, n2, m = 256, 512, 4
    a = torch.zeros((m, k), dtype=torch.float16, device="cuda")
    b = torch.zeros(k * n2 // 8, dtype=torch.int32, device="cuda")
    s = torch.ones((2, n2), dtype=torch.float16, device="cuda")
    h = torch.zeros((m, n2), dtype=torch.float16, device="cuda")
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
    for flags in (w4.W4A16_FLAG_SWIGLU | w4.W4A16_FLAG_GEGLU, w4.W4A16_FLAG_SWIGLU | FLAG_FORCE_MMA,
                  w4.W4A16_FLAG_GEGLU | w4.W4A16_FLAG_FORCE_SLICE):
        with pytest.raises(w4.W4A16Error) as e:
            w4.w4a16_gemm(a, b, h, s, None, None, None, ws, m, n2, k, 128, U4B8, flags)
        assert e.value.stage == 1 and e.value.detail == 4
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemm(a, b, h, s, None, None, None, ws, m, n2, k, 128, U4B8, w4.W4A16_FLAG_SWIGLU,
                      ldc=n2 // 2 - 8)
    assert e.value.stage == 1 and e.value.detail == 3


@pytest.mark.parametrize("kind", [1, 2])
def test_grouped_gated_matches_oracle(w4, orc, kind):
    """Experts' gate/up weights interleaved one by one; y[pair] = act(gate) * up of the pair's
    token with its expert.  The reference schedule is the oracle's CSR."""
    import torch
    n_exp, n_tok, top_k, k, n2, gs = 4, 100, 2, 512, 512, 128
    i = n2 // 2
    groups = k // gs
    seed = 6500 + kind
    sel = synth.routes(seed, n_tok, n_exp, top_k)
    a = synth.activations(seed, n_tok, k)
    qw = [synth.qweight(seed * 10 + e, k, n2) for e in range(n_exp)]
    s = [synth.scales(seed * 10 + e, groups, n2) for e in range(n_exp)]
    ex_ids, ex_off, ex_pairs, pair_tok = w4.w4a16_csr_from_token_routes(n_exp, n_tok, top_k, sel)
    n_pairs = n_tok * top_k
    per = k * n2 // 8
    b = torch.empty(n_exp * per, dtype=torch.int32, device="cuda")
    s_stack = torch.empty((n_exp * groups, n2), dtype=torch.float16, device="cuda")
    for e in range(n_exp):
        w4.w4_repack(interleave_on_device(w4, qw[e], n2), None, b[e * per:(e + 1) * per], k, n2)
        s_stack[e * groups:(e + 1) * groups] = interleave_on_device(w4, s[e], n2)
    flags = FLAG_IS_K_FULL | (w4.W4A16_FLAG_SWIGLU if kind == 1 else w4.W4A16_FLAG_GEGLU)
    ws = torch.zeros(w4.w4a16_grouped_workspace_size(n_pairs, len(ex_ids), n2, k, gs, flags),
                     dtype=torch.uint8, device="cuda")
    y = torch.full((n_pairs, i), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a16_gemm_grouped(torch_dev(a), b, y, s_stack, None, torch_dev(ex_ids), torch_dev(ex_off),
                          torch_dev(ex_pairs), torch_dev(pair_tok), len(ex_ids), n_exp, n_pairs,
                          n_tok, n2, k, gs, U4B8, flags, ws)
    torch.cuda.synchronize()
    assert w4.w4a16_status(ws) == 0
    got = y.float().cpu().numpy().astype(np.float64)
    ids, off, pairs, tok = orc.csr_from_token_routes(n_exp, n_tok, top_k, sel)
    g = np.zeros((n_pairs, i))
    u = np.zeros((n_pairs, i))
    for j, e in enumerate(ids):
        seg = pairs[off[j]:off[j + 1]]
        rows = np.ascontiguousarray(a[tok[seg]])
        g[seg] = orc.gemm(rows, np.ascontiguousarray(qw[e][:, :i]), np.ascontiguousarray(s[e][:, :i]),
                          None, None, gs, U4B8)
        u[seg] = orc.gemm(rows, np.ascontiguousarray(qw[e][:, i:]), np.ascontiguousarray(s[e][:, i:]),
                          None, None, gs, U4B8)
    glu_check(orc, got, g, u, kind)


@pytest.mark.parametrize("kind", [1, 2])
def test_gated_activation_at_extreme_gates(w4, orc, kind):
    """One-hot rows of A pick weight rows whose gate values run from -100 to 87.5 (codes 0..15
    at scale 12.5) and whose up values are 1, so the output is act(gate) itself: it must match
    the oracle and stay finite at both ends (for large negative gates the exponential in the
    sigmoid overflows to infinity, and the product must come out 0, not NaN)."""
    m, k, n2, gs = 16, 128, 512, 128
    i = n2 // 2
    codes = np.full((k, n2), 9, dtype=np.int64)             # up: (9 - 8) * 1 = 1
    for r in range(m):
        codes[r, :i] = (r + np.arange(i)) % 16              # every code in every row's columns
    qw = orc.pack_gptq(codes)
    s = np.ones((1, n2), dtype=np.float16)
    s[0, :i] = 12.5
    a = np.zeros((m, k), dtype=np.float16)
    a[np.arange(m), np.arange(m)] = 1.0
    got, _ = run_glu(w4, a, qw, s, None, k, n2, gs, U4B8, kind)
    g = (codes[:m, :i] - 8).astype(np.float64) * 12.5
    assert g.min() == -100.0 and g.max() == 87.5
    glu_check(orc, got, g, np.ones_like(g), kind)

"""BF16 activations (W4A16_FLAG_BF16) on the GPU against the oracle, through the C ABI.

A, scales, zeros and C are bfloat16; the codes and their tiles are the 4-bit ones of the fp16
path.  The oracle (gemm_bf16) reads the same bf16 bit patterns and sums exactly in double.

Tolerance.  The fp16 bar |c - ref| <= 1e-2 + 1e-2 |ref| covers a dequantised weight rounded
once to fp16 (unit roundoff 2^-11), fp32 sums and one rounding of C to fp16.  The bf16 path
has the same steps with unit roundoff 2^-8 for the weight and for C, eight times larger, so
its bar is the fp16 one scaled by 8: |c - ref| <= 8e-2 + 8e-2 |ref|.  Tests whose every
product and sum is exact (one nonzero weight per column) ask for equality.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import FLAG_ACT_ORDER, FLAG_HAS_ZP, FLAG_IS_K_FULL, U4, U4B8, torch_dev, within_tol

pytestmark = pytest.mark.gpu
RTOL = ATOL = 8e-2


@pytest.fixture(scope="module")
def w4():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import weight_only_int4_03_gb300 as w4
    return w4


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def dev16(bits):
    """A device int16 tensor of uint16 bit patterns (the library reads raw 16-bit words)."""
    return torch_dev(np.ascontiguousarray(bits).view(np.int16))


def out_values(c):
    """Doubles of a device int16 tensor of bf16 patterns."""
    u = c.cpu().numpy().view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def make(seed, m, k, n, gs, wt, act_order=False, sigma=1.0):
    groups = synth.group_count(k, gs)
    a = synth.bf16_bits(synth.Stream(seed, "A").normal(m * k, sigma)).reshape(m, k)
    qw = synth.qweight(seed, k, n)
    s = synth.bf16_bits(synth.scales(seed, groups, n).astype(np.float64))
    z = synth.bf16_bits(synth.zeros(seed, groups, n).astype(np.float64)) if wt == U4 else None
    perm = g_idx = None
    if act_order:
        perm = synth.permutation(seed, k)
        g_idx = synth.act_order_gidx(perm, gs if gs != -1 else k)
    return a, qw, s, z, g_idx, perm


def run_bf16(w4, a, qw, s, z, g_idx, perm, k, n, gs, wt, extra=0):
    import torch
    m = a.shape[0]
    b = torch.empty(k * n // 8, dtype=torch.int32, device="cuda")
    w4.w4_repack(torch_dev(qw), torch_dev(perm) if perm is not None else None, b, k, n)
    flags = FLAG_IS_K_FULL | w4.W4A16_FLAG_BF16 | extra
    flags |= FLAG_HAS_ZP if z is not None else 0
    flags |= FLAG_ACT_ORDER if perm is not None else 0
    glu = flags & (w4.W4A16_FLAG_SWIGLU | w4.W4A16_FLAG_GEGLU)
    ws = torch.zeros(w4.w4a16_workspace_size(m, n, k, gs, flags), dtype=torch.uint8, device="cuda")
    c = torch.full((m, n // 2 if glu else n), -1, dtype=torch.int16, device="cuda")  # NaN pattern
    w4.w4a16_gemm(dev16(a), b, c, dev16(s), dev16(z) if z is not None else None,
                  torch_dev(g_idx) if g_idx is not None else None,
                  torch_dev(perm) if perm is not None else None, ws, m, n, k, gs, wt, flags)
    torch.cuda.synchronize()
    assert w4.w4a16_status(ws) == 0
    return out_values(c)


@pytest.mark.parametrize("m,k,n,gs,wt,act", [
    (1, 1024, 512, 128, U4B8, False),      # one token: split tiles
    (16, 2048, 768, 128, U4, False),       # u4 zero points
    (64, 1024, 512, -1, U4B8, False),      # one group
    (40, 512, 1024, 32, U4, False),        # groups smaller than a 64-row block
    (300, 512, 1024, 64, U4B8, False),     # two token tiles
    (1000, 1024, 512, 128, U4B8, True),    # act-order (the gathered A is copied bit for bit)
    (4096, 256, 2048, 128, U4B8, False),   # paired token half-tiles, whole-tile epilogue
    (2000, 768, 2048, 128, U4, False),     # ragged token tail
])
def test_bf16_gemm_matches_oracle(w4, orc, m, k, n, gs, wt, act):
    seed = 9000 + m + k
    a, qw, s, z, g_idx, perm = make(seed, m, k, n, gs, wt, act, sigma=0.5 if wt == U4 else 1.0)
    got = run_bf16(w4, a, qw, s, z, g_idx, perm, k, n, gs, wt)
    ref = orc.gemm_bf16(a, qw, s, z, g_idx, gs, wt)
    ok, msg = within_tol(got, ref, RTOL, ATOL)
    assert ok, msg


@pytest.mark.parametrize("m", [3, 200])
def test_bf16_one_hot_is_bit_exact(w4, m):
    """Code 9 (weight 1 with zero point 8) at row pi(n) of column n, code 8 (weight 0)
    elsewhere, unit scales: C[:, n] = A[:, pi(n)] exactly in bf16."""
    k, n = 512, 256
    a = synth.bf16_bits(synth.Stream(9100 + m, "A").normal(m * k, 1.0)).reshape(m, k)
    pi = (np.arange(n) * 53 + 7) % k
    codes = np.full((k, n), 8, dtype=np.uint32)
    codes[pi, np.arange(n)] = 9
    qw = np.zeros((k // 8, n), dtype=np.uint32)
    for i in range(8):
        qw |= codes[i::8, :] << np.uint32(4 * i)
    s = synth.bf16_bits(np.ones((k // 128, n)))
    got = run_bf16(w4, a, qw.view(np.int32), s, None, None, None, k, n, 128, U4B8)
    want = (a[:, pi].astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kind", [1, 2])
def test_bf16_gated_matches_oracle(w4, orc, kind):
    """The gated epilogue in bf16: H = act(A Wg) * (A Wu), the gated bar of the fp16 tests with
    the GEMM bar tau scaled to 8e-2 + 8e-2 |x| and H rounded once to bf16."""
    m, k, n2, gs = 300, 512, 1024, 128
    i = n2 // 2
    a, qw, s, _, _, _ = make(9200 + kind, m, k, n2, gs, U4B8)
    import torch

    def inter(x):
        src = torch_dev(np.ascontiguousarray(x).view(np.int16) if x.dtype == np.uint16 else x)
        dst = torch.empty_like(src)
        w4.w4_gate_up_interleave(src, dst, x.shape[0], n2)
        return dst.cpu().numpy().view(x.dtype)

    flag = w4.W4A16_FLAG_SWIGLU if kind == 1 else w4.W4A16_FLAG_GEGLU
    got = run_bf16(w4, a, inter(qw), inter(s), None, None, None, k, n2, gs, U4B8, extra=flag)
    g = orc.gemm_bf16(a, np.ascontiguousarray(qw[:, :i]), np.ascontiguousarray(s[:, :i]), None, None, gs, U4B8)
    u = orc.gemm_bf16(a, np.ascontiguousarray(qw[:, i:]), np.ascontiguousarray(s[:, i:]), None, None, gs, U4B8)
    h = orc.glu(g, u, kind)
    act = orc.glu(g, np.ones_like(u), kind)
    tau_g = ATOL + RTOL * np.abs(g)
    tau_u = ATOL + RTOL * np.abs(u)
    bound = ATOL + RTOL * np.abs(h) + 1.2 * np.abs(u) * tau_g + np.abs(act) * tau_u + 1.2 * tau_g * tau_u
    assert np.all(np.isfinite(got))
    err = np.abs(got - h)
    assert np.all(err <= bound), f"{int((err > bound).sum())} outside, max err {err.max():.3e}"


def test_bf16_grouped_matches_oracle(w4, orc):
    """Grouped (expert-major CSR) bf16 GEMM; reference schedule from the oracle's CSR."""
    import torch
    n_exp, n_tok, top_k, k, n, gs = 4, 90, 2, 512, 512, 128
    groups = k // gs
    sel = synth.routes(9300, n_tok, n_exp, top_k)
    a = synth.bf16_bits(synth.Stream(9300, "A").normal(n_tok * k, 1.0)).reshape(n_tok, k)
    qws = [synth.qweight(9300 + e, k, n) for e in range(n_exp)]
    ss = [synth.bf16_bits(synth.scales(9300 + e, groups, n).astype(np.float64)) for e in range(n_exp)]
    ex_ids, ex_off, ex_pairs, pair_tok = w4.w4a16_csr_from_token_routes(n_exp, n_tok, top_k, sel)
    n_pairs = n_tok * top_k
    per = k * n // 8
    b = torch.empty(n_exp * per, dtype=torch.int32, device="cuda")
    for e in range(n_exp):
        w4.w4_repack(torch_dev(qws[e]), None, b[e * per:(e + 1) * per], k, n)
    flags = FLAG_IS_K_FULL | w4.W4A16_FLAG_BF16
    ws = torch.zeros(w4.w4a16_grouped_workspace_size(n_pairs, len(ex_ids), n, k, gs, flags),
                     dtype=torch.uint8, device="cuda")
    y = torch.full((n_pairs, n), -1, dtype=torch.int16, device="cuda")
    w4.w4a16_gemm_grouped(dev16(a), b, y, dev16(np.concatenate(ss)), None, torch_dev(ex_ids),
                          torch_dev(ex_off), torch_dev(ex_pairs), torch_dev(pair_tok), len(ex_ids),
                          n_exp, n_pairs, n_tok, n, k, gs, U4B8, flags, ws)
    torch.cuda.synchronize()
    assert w4.w4a16_status(ws) == 0
    got = out_values(y)
    ids, off, pairs, tok = orc.csr_from_token_routes(n_exp, n_tok, top_k, sel)
    ref = np.zeros_like(got)
    for j, e in enumerate(ids):
        seg = pairs[off[j]:off[j + 1]]
        ref[seg] = orc.gemm_bf16(np.ascontiguousarray(a[tok[seg]]), qws[e], ss[e], None, None, gs, U4B8)
    ok, msg = within_tol(got, ref, RTOL, ATOL)
    assert ok, msg


FORCE_MMA, FORCE_SLICE = 1 << 11, 1 << 13


@pytest.mark.parametrize("m,k,n,gs,wt,force", [
    (1, 1024, 512, 128, U4B8, FORCE_SLICE),
    (5, 4224, 768, 192, U4, FORCE_SLICE),       # groups straddle stages; partial last stage
    (16, 2048, 4096, -1, U4B8, FORCE_SLICE),
    (32, 1024, 512, 128, U4, FORCE_SLICE),      # four 8-token tiles
    (1, 2048, 512, 128, U4B8, FORCE_MMA),       # split-K, deferred group scales
    (16, 1024, 768, 256, U4, FORCE_MMA),
    (40, 2048, 512, 128, U4B8, FORCE_MMA),      # scales in the dequantisation, ragged tile
    (64, 1024, 1024, 64, U4, FORCE_MMA),
])
def test_bf16_small_m_kernels_match_oracle(w4, orc, m, k, n, gs, wt, force):
    seed = 9400 + m + k
    a, qw, s, z, g_idx, perm = make(seed, m, k, n, gs, wt, sigma=0.5 if wt == U4 else 1.0)
    got = run_bf16(w4, a, qw, s, z, g_idx, perm, k, n, gs, wt, extra=force)
    ref = orc.gemm_bf16(a, qw, s, z, g_idx, gs, wt)
    ok, msg = within_tol(got, ref, RTOL, ATOL)
    assert ok, msg


@pytest.mark.parametrize("force", [0, FORCE_MMA, FORCE_SLICE])
def test_bf16_one_hot_bit_exact_on_every_kernel(w4, force):
    """Code 9 at row pi(n), code 8 elsewhere, unit scales: C[:, n] = A[:, pi(n)] exactly,
    whichever kernel runs (default choice at M=4: the column-slice kernel)."""
    m, k, n = 4, 512, 256
    a = synth.bf16_bits(synth.Stream(9500, "A").normal(m * k, 1.0)).reshape(m, k)
    pi = (np.arange(n) * 29 + 3) % k
    codes = np.full((k, n), 8, dtype=np.uint32)
    codes[pi, np.arange(n)] = 9
    qw = np.zeros((k // 8, n), dtype=np.uint32)
    for i in range(8):
        qw |= codes[i::8, :] << np.uint32(4 * i)
    s = synth.bf16_bits(np.ones((k // 128, n)))
    got = run_bf16(w4, a, qw.view(np.int32), s, None, None, None, k, n, 128, U4B8, extra=force)
    want = (a[:, pi].astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("m,force", [(1, FORCE_SLICE), (8, FORCE_SLICE), (16, FORCE_SLICE),
                                     (8, FORCE_MMA), (16, FORCE_MMA), (8, 1 << 10)])
@pytest.mark.parametrize("wt", [U4B8, U4])
def test_bf16_one_hot_rows_give_rounded_weights_on_every_kernel(w4, orc, m, force, wt):
    """Row r of A is 1 at column k_r, so row r of C is row k_r of (q - z) s rounded once to
    bf16, bit for bit, with random codes, scales and zero points: the small-M kernels apply s to
    fp32 sums of the exact (q - z), the tcgen05 kernel rounds the product before its MMA.
    (q - z) s has at most 4 + 8 significant bits, so it is exact in float32 and synth.bf16_bits
    rounds it once.)"""
    k, n, gs = 256, 4096, 128
    _, qw, s, z, _, _ = make(9600 + m + (wt == U4), m, k, n, gs, wt)
    rows = (np.arange(m) * 37 + 5) % k
    a = np.zeros((m, k), dtype=np.uint16)
    a[np.arange(m), rows] = 0x3F80  # bf16 1.0
    got = run_bf16(w4, a, qw, s, z, None, None, k, n, gs, wt, extra=force)
    q = orc.unpack_gptq(qw, k, n).astype(np.float64)
    sd = orc.bf16_to_double(s)
    zd = orc.bf16_to_double(z) if z is not None else np.full_like(sd, 8.0)
    g = np.arange(k) // gs
    w = (q - zd[g]) * sd[g]
    want = (synth.bf16_bits(w[rows]).astype(np.uint32) << np.uint32(16)).view(np.float32)
    assert np.array_equal(got, want.astype(np.float64))

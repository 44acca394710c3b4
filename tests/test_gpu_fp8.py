"""FP8 E4M3 weights (W8A16) on the GPU against the oracle, through the C ABI.

Weights arrive as [K/4, N] words of four K-consecutive E4M3 codes (the pages' FP8 input ABI),
w8_repack turns them into the library's FP8 tiles, and W4A16_TYPE_FE4M3 GEMMs run the tcgen05
kernel.  Elementwise bar |c - ref| <= 1e-2 + 1e-2 |ref| (each code is exact in fp16; the product
with the scale is rounded once, as for the 4-bit types).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import (FLAG_ACT_ORDER, FLAG_FORCE_MMA, FLAG_FORCE_SLICE, FLAG_HAS_ZP, FLAG_IS_K_FULL,
                     torch_dev, within_tol)

pytestmark = pytest.mark.gpu
FE4M3 = 8


@pytest.fixture(scope="module")
def w4():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import weight_only_int4_03_gb300 as w4
    return w4


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def pack(codes):
    k, n = codes.shape
    c = codes.astype(np.uint32).reshape(k // 4, 4, n)
    w = np.zeros((k // 4, n), dtype=np.uint32)
    for i in range(4):
        w |= c[:, i, :] << np.uint32(8 * i)
    return w.view(np.int32)


def repack(w4, qw, k, n):
    import torch
    out = torch.empty(k * n // 4, dtype=torch.int32, device="cuda")
    w4.w8_repack(torch_dev(qw), out, k, n)
    return out


def run_fp8(w4, a, qw, s, k, n, gs, flags=FLAG_IS_K_FULL):
    import torch
    m = a.shape[0]
    b = repack(w4, qw, k, n)
    ws = torch.zeros(w4.w4a16_workspace_size(m, n, k, gs, flags), dtype=torch.uint8, device="cuda")
    c = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
    w4.w4a16_gemm(torch_dev(a), b, c, torch_dev(s), None, None, None, ws, m, n, k, gs, FE4M3, flags)
    torch.cuda.synchronize()
    assert w4.w4a16_status(ws) == 0
    return c.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("k,n", [(128, 256), (1024, 768), (4096, 4096)])
def test_fp8_repack_bit_exact_and_inverse(w4, orc, k, n):
    import torch
    qw = synth.fp8_weights(k + n, k, n)
    tiles = repack(w4, qw, k, n)
    assert np.array_equal(tiles.cpu().numpy(), orc.repack_fp8_tiles(qw, k, n))
    back = torch.empty((k // 4, n), dtype=torch.int32, device="cuda")
    w4.w8_unpack(tiles, back, k, n)
    assert np.array_equal(back.cpu().numpy(), qw)


@pytest.mark.parametrize("m,k,n,gs", [(1, 1024, 512, 128), (16, 2048, 768, 128), (64, 1024, 512, -1),
                                      (300, 512, 1024, 64), (1000, 1024, 512, 128),
                                      (4096, 256, 2048, 256)])
def test_fp8_gemm_matches_oracle(w4, orc, m, k, n, gs):
    seed = 8000 + m + k
    a = synth.activations(seed, m, k)
    qw = synth.fp8_weights(seed, k, n)
    s = synth.scales(seed, synth.group_count(k, gs), n, lo=1e-4, hi=2e-4)
    got = run_fp8(w4, a, qw, s, k, n, gs)
    ok, msg = within_tol(got, orc.gemm_fp8(a, qw, s, gs))
    assert ok, msg


@pytest.mark.parametrize("m,flags", [(40, FLAG_IS_K_FULL), (5, FLAG_IS_K_FULL | FLAG_FORCE_SLICE)])
def test_fp8_one_hot_is_bit_exact(w4, m, flags):
    """One 1.0 (0x38) per column at row pi(n), zeros elsewhere, unit scales: C[:, n] = A[:, pi(n)]
    exactly (one nonzero product, exact in fp32 and fp16); tcgen05 and column-slice kernels."""
    k, n = 512, 256
    a = synth.activations(8100 + m, m, k)
    pi = (np.arange(n) * 37 + 11) % k
    codes = np.zeros((k, n), dtype=np.uint8)
    codes[pi, np.arange(n)] = 0x38
    got = run_fp8(w4, a, pack(codes), np.ones((k // 128, n), dtype=np.float16), k, n, 128, flags)
    assert np.array_equal(got.astype(np.float16).view(np.uint16), a[:, pi].view(np.uint16))


@pytest.mark.parametrize("m,k,n,gs", [(1, 1024, 512, 128), (3, 4224, 768, 64), (8, 2048, 4096, -1),
                                      (16, 1024, 512, 256), (16, 4096, 4096, 128), (12, 4224, 768, 192)])
def test_fp8_column_slice_kernel_matches_oracle(w4, orc, m, k, n, gs):
    """FP8 tiles read through the column-slice view (four 256-byte rows per block)."""
    seed = 8600 + m + k
    a = synth.activations(seed, m, k)
    qw = synth.fp8_weights(seed, k, n)
    s = synth.scales(seed, synth.group_count(k, gs), n, lo=1e-4, hi=2e-4)
    got = run_fp8(w4, a, qw, s, k, n, gs, FLAG_IS_K_FULL | FLAG_FORCE_SLICE)
    ok, msg = within_tol(got, orc.gemm_fp8(a, qw, s, gs))
    assert ok, msg


def test_fp8_decode_shape_defaults_to_column_slice(w4):
    """M=4 at N=4096 (256 slices): the default choice is the column-slice kernel, the same bits
    as forcing it."""
    m, k, n = 4, 2048, 4096
    a = synth.activations(8700, m, k)
    qw = synth.fp8_weights(8700, k, n)
    s = synth.scales(8700, k // 128, n, lo=1e-4, hi=2e-4)
    d = run_fp8(w4, a, qw, s, k, n, 128)
    f = run_fp8(w4, a, qw, s, k, n, 128, FLAG_IS_K_FULL | FLAG_FORCE_SLICE)
    assert np.array_equal(d.astype(np.float16).view(np.uint16), f.astype(np.float16).view(np.uint16))


def test_fp8_nan_code_propagates(w4):
    """A NaN code (0x7F) in one column makes that column's outputs NaN and no other."""
    m, k, n = 8, 256, 256
    a = synth.activations(8200, m, k)
    codes = np.full((k, n), 0x30, dtype=np.uint8)   # 0.5
    codes[77, 5] = 0x7F
    got = run_fp8(w4, a, pack(codes), np.ones((2, n), dtype=np.float16), k, n, 128)
    assert np.all(np.isnan(got[:, 5]))
    assert np.all(np.isfinite(np.delete(got, 5, axis=1)))


def test_fp8_grouped_matches_oracle(w4, orc):
    import torch
    n_exp, n_tok, top_k, k, n, gs = 4, 60, 2, 512, 512, 128
    sel = synth.routes(8300, n_tok, n_exp, top_k)
    a = synth.activations(8300, n_tok, k)
    qws = [synth.fp8_weights(8300 + e, k, n) for e in range(n_exp)]
    ss = [synth.scales(8300 + e, k // gs, n, lo=1e-4, hi=2e-4) for e in range(n_exp)]
    ex_ids, ex_off, ex_pairs, pair_tok = w4.w4a16_csr_from_token_routes(n_exp, n_tok, top_k, sel)
    n_pairs = n_tok * top_k
    per = k * n // 4
    b = torch.empty(n_exp * per, dtype=torch.int32, device="cuda")
    for e in range(n_exp):
        b[e * per:(e + 1) * per] = repack(w4, qws[e], k, n)
    s_stack = torch_dev(np.concatenate(ss))
    ws = torch.zeros(w4.w4a16_grouped_workspace_size(n_pairs, len(ex_ids), n, k, gs, FLAG_IS_K_FULL),
                     dtype=torch.uint8, device="cuda")
    y = torch.empty((n_pairs, n), dtype=torch.float16, device="cuda")
    w4.w4a16_gemm_grouped(torch_dev(a), b, y, s_stack, None, torch_dev(ex_ids), torch_dev(ex_off),
                          torch_dev(ex_pairs), torch_dev(pair_tok), len(ex_ids), n_exp, n_pairs,
                          n_tok, n, k, gs, FE4M3, FLAG_IS_K_FULL, ws)
    torch.cuda.synchronize()
    assert w4.w4a16_status(ws) == 0
    got = y.float().cpu().numpy().astype(np.float64)
    ids, off, pairs, tok = orc.csr_from_token_routes(n_exp, n_tok, top_k, sel)
    ref = np.zeros_like(got)
    for i, e in enumerate(ids):
        seg = pairs[off[i]:off[i + 1]]
        ref[seg] = orc.gemm_fp8(np.ascontiguousarray(a[tok[seg]]), qws[e], ss[e], gs)
    ok, msg = within_tol(got, ref)
    assert ok, msg


def test_fp8_unsupported_combinations_rejected(w4):
    import torch
    m, k, n = 4, 256, 256
    a = torch.zeros((m, k), dtype=torch.float16, device="cuda")
    b = torch.zeros(k * n // 4, dtype=torch.int32, device="cuda")
    s = torch.ones((2, n), dtype=torch.float16, device="cuda")
    z = torch.full((2, n), 8.0, dtype=torch.float16, device="cuda")
    c = torch.zeros((m, n), dtype=torch.float16, device="cuda")
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
    g_idx = torch.zeros(k, dtype=torch.int32, device="cuda")
    perm = torch.arange(k, dtype=torch.int32, device="cuda")
    cases = [
        dict(zeros=z, flags=FLAG_HAS_ZP, detail=4),                 # no zero points for FP8
        dict(g_idx=g_idx, perm=perm, flags=FLAG_ACT_ORDER, detail=4),  # no act-order
        dict(flags=FLAG_FORCE_MMA, detail=4),                       # tcgen05 kernel only
        dict(gs=32, detail=7),                                      # groups of whole 64-row blocks
    ]
    big = torch.zeros((32, k), dtype=torch.float16, device="cuda")
    cbig = torch.zeros((32, n), dtype=torch.float16, device="cuda")
    with pytest.raises(w4.W4A16Error) as e:                          # FP8 slices: M <= 16
        w4.w4a16_gemm(big, b, cbig, s, None, None, None, ws, 32, n, k, 128, FE4M3,
                      FLAG_IS_K_FULL | FLAG_FORCE_SLICE)
    assert e.value.stage == 2 and e.value.detail == 3
    for cs in cases:
        with pytest.raises(w4.W4A16Error) as e:
            w4.w4a16_gemm(a, b, c, s, cs.get("zeros"), cs.get("g_idx"), cs.get("perm"), ws, m, n, k,
                          cs.get("gs", 128), FE4M3, cs.get("flags", 0))
        assert e.value.stage == 1 and e.value.detail == cs["detail"], cs


@pytest.mark.parametrize("m,flags", [(1, FLAG_IS_K_FULL | FLAG_FORCE_SLICE), (8, FLAG_IS_K_FULL | FLAG_FORCE_SLICE),
                                     (16, FLAG_IS_K_FULL | FLAG_FORCE_SLICE), (40, FLAG_IS_K_FULL)])
def test_fp8_one_hot_rows_give_rounded_weights(w4, orc, m, flags):
    """Row r of A is 1 at column k_r, so row r of C is row k_r of e4m3(code) s rounded once to
    fp16, bit for bit: the column-slice kernel applies s to fp32 sums of exact codes, the tcgen05
    kernel rounds the product before its MMA; both round the same exact value.  (A zero weight,
    code 0x80 being -0, meets the other rows' +0 products in the sum: zeros are compared by
    value, everything else by bits.)"""
    k, n, gs = 256, 4096, 128
    qw = synth.fp8_weights(8200 + m, k, n)
    s = synth.scales(8200 + m, k // gs, n)
    rows = (np.arange(m) * 37 + 5) % k
    a = np.zeros((m, k), dtype=np.float16)
    a[np.arange(m), rows] = 1.0
    got = run_fp8(w4, a, qw, s, k, n, gs, flags)
    want = orc.dequant_fp8(qw, s, k, n, gs)[rows].astype(np.float16)
    got16 = got.astype(np.float16)
    nz = want != 0
    assert np.all(got16[~nz] == 0)
    assert np.array_equal(got16[nz].view(np.uint16), want[nz].view(np.uint16))

"""CUDA path vs the CPU oracle, through the C ABI (needs a GB300 and the built library)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import (ATOL, FLAG_A_SMEM, FLAG_FORCE_MMA, FLAG_FORCE_SIMT, FLAG_FORCE_SLICE, FLAG_FORCE_TC,
                     FLAG_STATIC_WEIGHTS, RTOL, U4, U4B8, DeviceProblem, make_problem,
                     oracle_ref, repack_device, torch_dev, within_tol)

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


def check(dp, orc, rows=None):
    got = dp.result()
    if rows is not None:
        got = got[rows]
    ok, msg = within_tol(got, oracle_ref(orc, dp.pb, rows))
    assert ok, msg
    assert dp.status() == 0


# --- layout ----------------------------------------------------------------------------------

@pytest.mark.parametrize("k,n,with_perm", [(128, 256, False), (256, 512, False), (256, 512, True),
                                           (1024, 768, True), (4096, 4096, False)])
def test_repack_matches_oracle_bit_exact(w4, orc, k, n, with_perm):
    qw = synth.qweight(k + n, k, n)
    perm = synth.permutation(k, k) if with_perm else None
    out = repack_device(w4, qw, perm, k, n).cpu().numpy()
    assert np.array_equal(out, orc.repack_tiles(qw, perm, k, n))


@pytest.mark.parametrize("k,n", [(128, 256), (512, 1024), (4096, 12288)])
def test_unpack_inverts_repack(w4, k, n):
    import torch
    qw = synth.qweight(7 * k + n, k, n)
    tiles = repack_device(w4, qw, None, k, n)
    back = torch.empty((k // 8, n), dtype=torch.int32, device="cuda")
    w4.w4_unpack(tiles, back, k, n)
    assert np.array_equal(back.cpu().numpy(), qw)


def test_repack_reports_out_of_range_perm(w4):
    import torch
    k, n = 128, 256
    qw = synth.qweight(3, k, n)
    perm = np.arange(k, dtype=np.int32)
    perm[5] = k + 7
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(k * n // 8, dtype=torch.int32, device="cuda")
    w4.w4_repack(torch_dev(qw), torch_dev(perm), out, k, n, status=status)
    assert int(status.item()) & w4.W4A16_DEV_PERM


# --- GEMM parity -------------------------------------------------------------------------------

def test_tiny_config(w4, orc):
    """M=16, K=256, N=256, group 128, u4b8, seed 0 (the tiny workload) -- every element."""
    dp = DeviceProblem(w4, make_problem(0, 16, 256, 256))
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("m", [1, 3, 16, 17, 32, 33, 64, 100, 128, 200, 256, 257, 300, 600, 1000, 1500])
def test_m_sweep_u4b8(w4, orc, m):
    """Ragged M across token tiles; K=512 (8 row blocks), N=512 (4 column tiles): stream-K splits."""
    dp = DeviceProblem(w4, make_problem(100 + m, m, 512, 512))
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("gs", [16, 32, 64, 128, 256, -1])
def test_group_sizes(w4, orc, gs):
    dp = DeviceProblem(w4, make_problem(200 + max(gs, 0), 20, 512, 256, group_size=gs))
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("m", [1, 16, 100, 300])
def test_zero_points_u4(w4, orc, m):
    dp = DeviceProblem(w4, make_problem(300 + m, m, 768, 512, weight_type=U4, sigma=0.5))
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("m,gs", [(1, 128), (16, 128), (200, 64), (33, 32), (1000, 128), (64, 128)])
def test_act_order(w4, orc, m, gs):
    dp = DeviceProblem(w4, make_problem(400 + m, m, 1024, 512, group_size=gs, act_order=True))
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("flag", [FLAG_A_SMEM, FLAG_FORCE_SIMT])
@pytest.mark.parametrize("m", [1, 40, 300])
def test_alternate_paths(w4, orc, flag, m):
    """Dequantised weights staged in shared memory, and the CUDA-core reference kernel."""
    dp = DeviceProblem(w4, make_problem(500 + m, m, 512, 512, weight_type=U4), flags_extra=flag)
    dp.run()
    check(dp, orc)


# --- the two kernels: small-M register-fragment kernel and tcgen05 kernel, each forced -------

@pytest.mark.parametrize("flag", [FLAG_FORCE_MMA, FLAG_FORCE_TC])
@pytest.mark.parametrize("m", [1, 2, 5, 8, 9, 15, 16, 24, 31, 32, 33, 48, 63, 64])
def test_small_m_both_kernels(w4, orc, flag, m):
    """Every small M through both kernels; K=1024 (16 row blocks, 2 stages), N=768 (6 column
    tiles, so stream-K splits tiles over several CTAs)."""
    dp = DeviceProblem(w4, make_problem(1000 + m, m, 1024, 768), flags_extra=flag)
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("gs", [16, 32, 64, 128, 512, -1])
@pytest.mark.parametrize("m", [1, 8, 40])
def test_small_m_kernel_group_sizes(w4, orc, gs, m):
    dp = DeviceProblem(w4, make_problem(1100 + m + max(gs, 0), m, 1024, 512, group_size=gs),
                       flags_extra=FLAG_FORCE_MMA)
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("gs", [-1, 2112])
@pytest.mark.parametrize("m", [1, 16])
def test_small_m_kernel_long_groups(w4, orc, gs, m):
    """Groups of more than 32 blocks (one group over K = 4224, or two of 33 blocks): the group
    end is found by count, not by the per-stage mask, and split segments of a block or two end
    inside a group, so each adds its share of the group's scaled sum."""
    dp = DeviceProblem(w4, make_problem(1150 + m + max(gs, 0), m, 4224, 512, group_size=gs),
                       flags_extra=FLAG_FORCE_MMA)
    dp.run()
    check(dp, orc)


# --- column-slice small-M kernel (16-column slices over all of K, no split-K) ----------------

@pytest.mark.parametrize("m,k,n,gs,kw", [
    (1, 1024, 256, 128, {}),                                  # 2 stages of 8 blocks, 16 slices
    (3, 2048, 512, -1, {}),                                   # one group over K
    (8, 4224, 512, 64, {}),                                   # 66 blocks: last stage has 2
    (9, 1536, 256, 512, dict(weight_type=U4, sigma=0.5)),     # u4 zeros, one group per stage
    (16, 4224, 768, 192, dict(weight_type=U4, sigma=0.5)),    # groups straddle stages
    (16, 4096, 4096, 128, {}),                                # 256 slices: one per CTA
    (5, 4096, 12288, 128, {}),                                # 768 slices: 3 per CTA
    (24, 4224, 768, 192, dict(weight_type=U4, sigma=0.5)),    # four 8-token tiles, ragged
    (32, 4096, 4096, 128, {}),                                # four full tiles, 256 slices
    (17, 1024, 256, -1, {}),
])
def test_slice_kernel(w4, orc, m, k, n, gs, kw):
    dp = DeviceProblem(w4, make_problem(1500 + m + k % 997, m, k, n, group_size=gs, **kw),
                       flags_extra=FLAG_FORCE_SLICE)
    dp.run()
    rows = None if m * n <= 32 * 4096 else [0, m - 1]
    check(dp, orc, rows)


@pytest.mark.parametrize("m,gs", [(1, 128), (16, 64)])
def test_slice_kernel_act_order(w4, orc, m, gs):
    dp = DeviceProblem(w4, make_problem(1600 + m, m, 2048, 512, group_size=gs, act_order=True),
                       flags_extra=FLAG_FORCE_SLICE)
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("m", [1, 16])
def test_slice_kernel_repeatable_and_static_weights(w4, m):
    """Fixed-order cross-warp sums: repeated calls are bit-identical, with or without the
    static-weights flag (weights read before the preceding kernel finishes)."""
    pb = make_problem(1700 + m, m, 4096, 4096)
    dp = DeviceProblem(w4, pb, flags_extra=FLAG_FORCE_SLICE)
    dp.run()
    first = dp.c.cpu().numpy().copy()
    ds = DeviceProblem(w4, pb, flags_extra=FLAG_FORCE_SLICE | FLAG_STATIC_WEIGHTS)
    for _ in range(3):
        dp.run()
        ds.run()
        assert np.array_equal(dp.c.cpu().numpy().view(np.uint16), first.view(np.uint16))
        assert np.array_equal(ds.c.cpu().numpy().view(np.uint16), first.view(np.uint16))
    assert dp.status() == 0 and ds.status() == 0


def test_slice_kernel_is_the_default_for_decode_shapes(w4):
    """M <= 16 with whole-block groups and at least one slice per SM goes to the column-slice
    kernel by default: the same bits as forcing it."""
    pb = make_problem(1800, 4, 4096, 4096)
    d0 = DeviceProblem(w4, pb)
    d1 = DeviceProblem(w4, pb, flags_extra=FLAG_FORCE_SLICE)
    d0.run()
    d1.run()
    assert np.array_equal(d0.c.cpu().numpy().view(np.uint16), d1.c.cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("m", [1, 7, 16, 64])
def test_small_m_kernel_zero_points(w4, orc, m):
    dp = DeviceProblem(w4, make_problem(1200 + m, m, 768, 512, weight_type=U4, sigma=0.5),
                       flags_extra=FLAG_FORCE_MMA)
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("m,gs", [(1, 128), (8, 32), (33, 64)])
def test_small_m_kernel_act_order(w4, orc, m, gs):
    dp = DeviceProblem(w4, make_problem(1300 + m, m, 1024, 512, group_size=gs, act_order=True),
                       flags_extra=FLAG_FORCE_MMA)
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("m", [1, 8, 16, 64])
def test_small_m_kernel_repeatable(w4, m):
    dp = DeviceProblem(w4, make_problem(1400 + m, m, 2048, 1024), flags_extra=FLAG_FORCE_MMA)
    dp.run()
    first = dp.c.cpu().numpy().copy()
    for _ in range(3):
        dp.run()
        assert np.array_equal(dp.c.cpu().numpy().view(np.uint16), first.view(np.uint16))


@pytest.mark.parametrize("m,k,n,kw", [(1, 4096, 4096, {}), (16, 1024, 768, dict(weight_type=U4, sigma=0.5)),
                                      (8, 2048, 512, dict(act_order=True)), (300, 512, 512, {})])
def test_static_weights_flag(w4, orc, m, k, n, kw):
    """Weights read before the preceding kernel completes: same results, several calls in a row
    (the stages issued early wrap around the ring)."""
    pb = make_problem(1600 + m, m, k, n, **kw)
    dp = DeviceProblem(w4, pb, flags_extra=FLAG_STATIC_WEIGHTS)
    for _ in range(3):
        dp.run()
    check(dp, orc)
    plain = DeviceProblem(w4, pb)
    plain.run()
    import torch
    torch.cuda.synchronize()
    assert np.array_equal(dp.c.cpu().numpy().view(np.uint16), plain.c.cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("m,k,n,flag", [(1, 4096, 4096, 0), (13, 4224, 4096, 0), (5, 1152, 12288, 0),
                                        (64, 4096, 4096, FLAG_FORCE_TC), (40, 2176, 4096, FLAG_FORCE_MMA)])
def test_tile_aligned_split_schedule(w4, orc, m, k, n, flag):
    """Shapes whose tiles x CTAs-per-tile cover most of the GPU run one near-equal K-range per
    CTA (uneven when the split does not divide the 64-row blocks: 66 blocks over 9, 18 over 3)."""
    dp = DeviceProblem(w4, make_problem(1700 + m, m, k, n), flags_extra=flag)
    for _ in range(2):
        dp.run()
    check(dp, orc)


def test_kernel_flags_rejected(w4):
    pb = make_problem(1500, 65, 256, 256)
    dp = DeviceProblem(w4, pb, flags_extra=FLAG_FORCE_MMA)
    with pytest.raises(w4.W4A16Error) as e:
        dp.run()
    assert e.value.stage == 2
    dp = DeviceProblem(w4, make_problem(1501, 4, 256, 256), flags_extra=FLAG_FORCE_MMA | FLAG_FORCE_TC)
    with pytest.raises(w4.W4A16Error) as e:
        dp.run()
    assert e.value.stage == 1 and e.value.detail == 4


def test_large_k_many_tiles(w4, orc):
    """K=4096, N=4096, M=1000: four token tiles, 32 column tiles, 64 row blocks."""
    dp = DeviceProblem(w4, make_problem(601, 1000, 4096, 4096))
    dp.run()
    rows = [0, 1, 255, 256, 511, 512, 767, 768, 999]
    check(dp, orc, rows)


# --- exact pins ---------------------------------------------------------------------------------

def _const_codes(orc, k, n, value):
    return orc.pack_gptq(np.full((k, n), value, dtype=np.uint8))


def test_code8_gives_positive_zero(w4, orc):
    pb = make_problem(701, 37, 512, 512)
    pb.qweight = _const_codes(orc, 512, 512, 8)
    dp = DeviceProblem(w4, pb)
    dp.run()
    import torch
    torch.cuda.synchronize()
    assert int(dp.c.view(torch.int16).abs().max().item()) == 0


@pytest.mark.parametrize("m", [1, 24, 300])
def test_one_hot_is_bit_exact(w4, orc, m):
    k, n = 512, 512
    pb = make_problem(702 + m, m, k, n)
    pi = (np.arange(n) * 37 + 11) % k
    codes = np.full((k, n), 8, dtype=np.uint8)
    codes[pi, np.arange(n)] = 9
    pb.qweight = orc.pack_gptq(codes)
    pb.scales = np.ones_like(pb.scales)
    dp = DeviceProblem(w4, pb)
    dp.run()
    got = dp.c.cpu().numpy()
    assert np.array_equal(got.view(np.uint16), pb.a[:, pi].view(np.uint16))


def test_zero_point_eight_matches_u4b8_bit_exact(w4):
    pb = make_problem(703, 77, 512, 512)
    d1 = DeviceProblem(w4, pb)
    d1.run()
    pb2 = make_problem(703, 77, 512, 512)
    pb2.weight_type = U4
    pb2.zeros = np.full_like(pb2.scales, 8)
    d2 = DeviceProblem(w4, pb2)
    d2.run()
    assert np.array_equal(d1.c.cpu().numpy().view(np.uint16), d2.c.cpu().numpy().view(np.uint16))


def test_identity_act_order_matches_plain_bit_exact(w4):
    pb = make_problem(704, 50, 512, 512)
    d1 = DeviceProblem(w4, pb)
    d1.run()
    pb2 = make_problem(704, 50, 512, 512)
    pb2.perm = np.arange(512, dtype=np.int32)
    pb2.g_idx = (np.arange(512) // 128).astype(np.int32)
    d2 = DeviceProblem(w4, pb2)
    d2.run()
    assert np.array_equal(d1.c.cpu().numpy().view(np.uint16), d2.c.cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("m", [1, 64, 700])
def test_repeated_runs_bit_identical(w4, m):
    dp = DeviceProblem(w4, make_problem(705 + m, m, 2048, 1024))
    dp.run()
    first = dp.c.cpu().numpy().copy()
    for _ in range(3):
        dp.run()
        assert np.array_equal(dp.c.cpu().numpy().view(np.uint16), first.view(np.uint16))


@pytest.mark.parametrize("m", [8, 300])   # element-wise and row-staged gathers
def test_unequal_groups_reported(w4, m):
    pb = make_problem(706, m, 256, 256, act_order=True)
    pb.g_idx = pb.g_idx.copy()
    pb.g_idx[pb.perm[0]] = 1   # sorted row 0 claims group 1
    dp = DeviceProblem(w4, pb)
    dp.run()
    assert dp.status() & w4.W4A16_DEV_GIDX


# --- edges ----------------------------------------------------------------------------------

def test_empty_m_is_a_noop(w4):
    import torch
    pb = make_problem(800, 1, 256, 256)
    dp = DeviceProblem(w4, pb)
    dp.c.fill_(3.0)
    w4.w4a16_gemm(dp.a, dp.b, dp.c, dp.scales, None, None, None, dp.ws, 0, 256, 256, 128, U4B8, 0)
    torch.cuda.synchronize()
    assert float(dp.c.float().min()) == 3.0


@pytest.mark.parametrize("m,flag", [(45, 0), (5, FLAG_FORCE_SLICE), (12, FLAG_FORCE_MMA)])
def test_strided_a_and_c(w4, orc, m, flag):
    """lda > K and ldc > N through each kernel; the columns of C past N stay untouched."""
    import torch
    pb = make_problem(801 + m, m, 512, 256)
    dp = DeviceProblem(w4, pb, flags_extra=flag)
    lda, ldc = 512 + 24, 256 + 40
    a_big = torch.zeros((pb.m, lda), dtype=torch.float16, device="cuda")
    a_big[:, :512] = dp.a
    c_big = torch.full((pb.m, ldc), 7.0, dtype=torch.float16, device="cuda")
    w4.w4a16_gemm(a_big, dp.b, c_big, dp.scales, None, None, None, dp.ws, pb.m, 256, 512, 128, U4B8,
                  dp.flags, lda=lda, ldc=ldc)
    torch.cuda.synchronize()
    got = c_big[:, :256].float().cpu().numpy().astype(np.float64)
    ok, msg = within_tol(got, oracle_ref(orc, pb))
    assert ok, msg
    assert float(c_big[:, 256:].float().min()) == 7.0 and float(c_big[:, 256:].float().max()) == 7.0


def test_argument_errors_raise(w4):
    pb = make_problem(802, 4, 256, 256)
    dp = DeviceProblem(w4, pb)
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemm(dp.a, dp.b, dp.c, dp.scales, None, None, None, dp.ws, 4, 256, 256, 100, U4B8, 0)
    assert e.value.stage == 1
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemm(dp.a, dp.b, dp.c, dp.scales, None, None, None, dp.ws, 4, 256, 256, 128, U4B8, 0,
                      workspace_bytes=64)
    assert e.value.stage == 1 and e.value.detail == 6


def test_bounded_wait_selftest_keeps_context_usable(w4, orc):
    import torch
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    w4.w4a16_selftest_timeout(ws, 20_000_000)
    assert w4.w4a16_status(ws) & w4.W4A16_DEV_TIMEOUT
    assert w4.w4a16_status(ws) == 0
    dp = DeviceProblem(w4, make_problem(803, 5, 256, 256))
    dp.run()
    check(dp, orc)


# --- grouped (MoE) ------------------------------------------------------------------------------

def _grouped_problem(seed, n_exp, n_tok, top_k, k, n, weight_type=U4B8, gs=128):
    groups = synth.group_count(k, gs)
    sel = synth.routes(seed, n_tok, n_exp, top_k)
    a = synth.activations(seed, n_tok, k)
    qw = synth.qweight(seed, k, n * n_exp).reshape(k // 8, n_exp, n).transpose(1, 0, 2).copy()
    s = synth.scales(seed, n_exp * groups, n).reshape(n_exp, groups, n)
    z = synth.zeros(seed, n_exp * groups, n).reshape(n_exp, groups, n) if weight_type == U4 else None
    return sel, a, qw, s, z


def run_grouped(w4, sel, a, qw, s, z, n_exp, n_tok, top_k, k, n, weight_type=U4B8, gs=128):
    import torch
    ex_ids, ex_off, ex_pairs, pair_tok = w4.w4a16_csr_from_token_routes(n_exp, n_tok, top_k, sel)
    n_pairs = n_tok * top_k
    b = torch.empty(n_exp * k * n // 8, dtype=torch.int32, device="cuda")
    for e in range(n_exp):
        w4.w4_repack(torch_dev(qw[e]), None, b[e * k * n // 8:(e + 1) * k * n // 8], k, n)
    flags = (1 << 2) | ((1 << 3) if z is not None else 0)
    ws = torch.zeros(w4.w4a16_grouped_workspace_size(n_pairs, len(ex_ids), n, k, gs, flags),
                     dtype=torch.uint8, device="cuda")
    y = torch.empty((n_pairs, n), dtype=torch.float16, device="cuda")
    w4.w4a16_gemm_grouped(torch_dev(a), b, y, torch_dev(s), torch_dev(z) if z is not None else None,
                          torch_dev(ex_ids), torch_dev(ex_off), torch_dev(ex_pairs), torch_dev(pair_tok),
                          len(ex_ids), n_exp, n_pairs, n_tok, n, k, gs, weight_type, flags, ws)
    torch.cuda.synchronize()
    assert w4.w4a16_status(ws) == 0
    return y.float().cpu().numpy().astype(np.float64), (ex_ids, ex_off, ex_pairs, pair_tok)


@pytest.mark.parametrize("n_exp,n_tok,top_k,wt", [(4, 32, 2, U4B8), (8, 100, 2, U4), (3, 300, 1, U4B8)])
def test_grouped_small(w4, orc, n_exp, n_tok, top_k, wt):
    k, n = 256, 512
    sel, a, qw, s, z = _grouped_problem(900 + n_tok, n_exp, n_tok, top_k, k, n, wt)
    y, csr = run_grouped(w4, sel, a, qw, s, z, n_exp, n_tok, top_k, k, n, wt)
    # The reference schedule comes from the oracle's own CSR builder.
    csr_ref = orc.csr_from_token_routes(n_exp, n_tok, top_k, sel)
    ref = orc.grouped(a, qw.ravel(), s, z, *csr_ref, k, n, 128, wt)
    ok, msg = within_tol(y, ref)
    assert ok, msg


def test_grouped_segment_equals_dense(w4):
    """Every expert segment equals a dense call on its gathered rows up to fp32 summation order
    (the two calls split K differently): at most one fp16 rounding step apart."""
    import torch
    n_exp, n_tok, top_k, k, n = 4, 40, 2, 512, 256
    sel, a, qw, s, z = _grouped_problem(950, n_exp, n_tok, top_k, k, n)
    y, (ex_ids, ex_off, ex_pairs, pair_tok) = run_grouped(w4, sel, a, qw, s, z, n_exp, n_tok, top_k, k, n)
    for i, e in enumerate(ex_ids):
        pairs = ex_pairs[ex_off[i]:ex_off[i + 1]]
        rows = a[pair_tok[pairs]]
        pb = make_problem(0, len(pairs), k, n)
        pb.a, pb.qweight, pb.scales = rows, qw[e], s[e]
        dp = DeviceProblem(w4, pb)
        dp.run()
        dense = dp.result()
        assert np.all(np.abs(dense - y[pairs]) <= 1e-3 * np.abs(dense) + 1e-3)


# --- loader helpers and workspace recovery --------------------------------------------------

def test_zero_points_check(w4):
    """Integer zero points in [0, 15] pass; a fraction, 16, a negative value or NaN anywhere
    is reported."""
    import torch
    good = torch.tensor([[0, 1, 7, 15]], dtype=torch.float16, device="cuda").repeat(300, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    w4.w4a16_zero_points_check(good, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for bad in (7.5, 16.0, -1.0, float("nan"), 0.0625):
        z = good.clone()
        z[123, 2] = bad
        status.zero_()
        w4.w4a16_zero_points_check(z, status)
        torch.cuda.synchronize()
        assert int(status.item()) & w4.W4A16_DEV_ZERO, bad


def test_converted_qzeros_run_as_u4(w4, orc):
    """Packed GPTQ zero words converted by the library's loader helper (code + 1) drive a u4
    GEMM that matches the oracle fed with the oracle's own conversion."""
    m, k, n, gs = 9, 512, 256, 128
    pb = make_problem(805, m, k, n, weight_type=U4)
    groups = k // gs
    codes = np.asarray(synth.qweight(806, 8 * groups, n)).view(np.uint32)[:groups, : n // 8]
    codes = codes & np.uint32(0x77777777)   # stored codes 0..7: zero points 1..8
    qz = np.ascontiguousarray(codes).view(np.int32)
    pb.zeros = w4.w4_qzeros_to_zero_points(qz, groups, n)
    ref_z = orc.qzeros_to_zero_points(qz, groups, n)
    assert np.array_equal(pb.zeros.astype(np.float64), ref_z)
    dp = DeviceProblem(w4, pb)
    dp.run()
    check(dp, orc)


def test_workspace_reset_after_timeout_report(w4, orc):
    """The recovery documented for W4A16_DEV_TIMEOUT: a workspace whose counters were left
    part-way (simulated here by writing them on the host side) and whose status word holds the
    bit is read back, zero-filled again, and the next call is correct."""
    import torch
    pb = make_problem(807, 8, 4096, 512)   # few tiles, many CTAs per tile: split tiles
    dp = DeviceProblem(w4, pb, flags_extra=FLAG_FORCE_MMA)
    dp.ws.fill_(3)                          # counters 0x03030303, partials garbage
    dp.ws[:4].copy_(torch.tensor([w4.W4A16_DEV_TIMEOUT], dtype=torch.int32).view(torch.uint8))
    assert w4.w4a16_status(dp.ws) & w4.W4A16_DEV_TIMEOUT
    dp.ws.zero_()                           # the recovery step
    dp.run()
    check(dp, orc)


@pytest.mark.parametrize("m,flag", [(1, FLAG_FORCE_SLICE), (8, FLAG_FORCE_SLICE), (16, FLAG_FORCE_SLICE),
                                    (8, FLAG_FORCE_MMA), (16, FLAG_FORCE_MMA), (8, FLAG_FORCE_TC)])
@pytest.mark.parametrize("wt", [U4B8, U4])
def test_one_hot_rows_give_rounded_weights_on_every_kernel(w4, orc, m, flag, wt):
    """Row r of A is 1 at column k_r and 0 elsewhere, so row r of C is row k_r of the
    dequantised weight, (q - z) s, rounded once to fp16: bit for bit on every kernel, whether it
    rounds (q - z) s to fp16 before the MMA or applies s to fp32 sums afterwards."""
    k, n = 256, 4096  # N / 16 >= the SM count: the column-slice kernel takes these shapes
    pb = make_problem(7100 + m + (wt == U4), m, k, n, weight_type=wt)
    rows = (np.arange(m) * 37 + 5) % k
    a = np.zeros((m, k), dtype=np.float16)
    a[np.arange(m), rows] = 1.0
    pb.a = a
    dp = DeviceProblem(w4, pb, flags_extra=flag)
    dp.run()
    got = dp.result()
    w = orc.dequant(pb.qweight, pb.scales, pb.zeros, None, k, n, pb.group_size, wt)
    want = w[rows].astype(np.float16)
    assert dp.status() == 0
    assert np.array_equal(got.astype(np.float16).view(np.uint16), want.view(np.uint16))

"""Pins for the CPU oracle: facts fixed by the pages or by the mathematics, not by the oracle.

Each `pin_*` function takes an `oracle.Oracle` and returns None when the oracle satisfies the
fact, or a short message describing the violation.  tests/test_oracle_pins.py runs every pin
against the real oracle; tests/test_oracle_mutations.py compiles copies of the oracle with a
planted mistake and checks that some pin catches each one.

Shapes are non-square on purpose (M != K != N, several groups) so that a transposed operand
or a swapped index cannot pass a closed form by symmetry.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U4, U4B8 = 4, 5


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _codes_const(orc, k, n, value):
    return orc.pack_gptq(np.full((k, n), value, dtype=np.uint8))


def _rowsums(a16: np.ndarray, weights=None) -> np.ndarray:
    """Exact (fsum) sums over k of A[m][k] * weights[k] in double."""
    a = a16.astype(np.float64)
    if weights is None:
        weights = np.ones(a.shape[1])
    return np.array([math.fsum(a[i] * weights) for i in range(a.shape[0])])


def _mismatch(name, got, want, rtol=0.0, atol=0.0):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if got.shape != want.shape:
        return f"{name}: shape {got.shape} != {want.shape}"
    with np.errstate(invalid="ignore"):
        bad = ~((got == want) | (np.abs(got - want) <= atol + rtol * np.abs(want)))
    if bad.any():
        idx = np.argwhere(bad)[0]
        return f"{name}: first mismatch at {tuple(idx)}: {got[tuple(idx)]!r} vs {want[tuple(idx)]!r}"
    return None


# --- binary16 -----------------------------------------------------------------------------

def pin_half_decode_all_patterns(orc):
    """Every binary16 bit pattern decodes as numpy's float16 does (a library routine)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.half_to_double(bits.view(np.float16))
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    if not np.array_equal(np.isnan(got), nan):
        return "half decode: NaN patterns differ"
    return _mismatch("half decode", got[~nan], want[~nan])


# --- GPTQ packing -------------------------------------------------------------------------

def pin_nibble_order_low_first(orc):
    """Word 0x76543210 holds codes 0..7 for rows 0..7 (row 8r+i at bits 4i)."""
    qw = np.array([[0x76543210]], dtype=np.uint32).view(np.int32)
    got = orc.unpack_gptq(qw, 8, 1)[:, 0]
    return _mismatch("nibble order", got, np.arange(8))


def pin_pack_unpack_brute_force(orc):
    """q[k][n] = (k + 3n) mod 16 survives pack -> unpack; packed words match a per-bit build."""
    k, n = 48, 5
    codes = ((np.arange(k)[:, None] + 3 * np.arange(n)[None, :]) % 16).astype(np.uint8)
    words = orc.pack_gptq(codes)
    for r in range(k // 8):
        for c in range(n):
            want = sum(int(codes[8 * r + i, c]) << (4 * i) for i in range(8))
            got = int(words[r, c]) & 0xFFFFFFFF
            if got != want:
                return f"pack: word ({r},{c}) = {got:#x}, want {want:#x}"
    return _mismatch("unpack", orc.unpack_gptq(words, k, n), codes)


def pin_unpack_random_words(orc):
    """Unpacking random words and repacking gives the same words (all 2^32 values reachable)."""
    qw = synth.qweight(11, 64, 24)
    codes = orc.unpack_gptq(qw, 64, 24)
    if codes.max() > 15:
        return "unpack: code above 15"
    back = orc.pack_gptq(codes)
    if not np.array_equal(back, qw):
        return "pack(unpack(x)) != x"
    return None


# --- dequant and GEMM ---------------------------------------------------------------------

def pin_hand_worked_example(orc):
    g = _golden("hand_worked_example.json")
    qw = np.array(g["qweight_words"], dtype=np.uint32).view(np.int32)
    s = np.array(g["scales"], dtype=np.float16)
    a = np.array(g["a"], dtype=np.float16)
    got = orc.gemm(a, qw, s, group_size=g["group_size"], weight_type=U4B8, threads=1)
    return _mismatch("hand example", got, np.array(g["c"], dtype=np.float64))


def pin_code8_gives_exact_zero(orc):
    """u4b8 code 8 is weight 0: C == +0 exactly for any A and scales."""
    m, k, n = 3, 256, 40
    a = synth.activations(1, m, k)
    s = synth.scales(2, 2, n)
    got = orc.gemm(a, _codes_const(orc, k, n, 8), s, group_size=128, weight_type=U4B8)
    if np.any(got != 0.0) or np.any(np.signbit(got)):
        return "q=8 did not give +0"
    return None


def pin_code0_unit_scale_closed_form(orc):
    """u4b8, q = 0, s = 1: C[m][n] = -8 * sum_k A[m][k] for every n."""
    m, k, n = 5, 384, 24
    a = synth.activations(3, m, k)
    s = np.ones((3, n), dtype=np.float16)
    got = orc.gemm(a, _codes_const(orc, k, n, 0), s, group_size=128, weight_type=U4B8)
    want = np.repeat((-8.0 * _rowsums(a))[:, None], n, axis=1)
    return _mismatch("q=0 closed form", got, want, rtol=1e-13, atol=1e-12)


def pin_group_boundaries(orc):
    """q = 9 (weight = s) and s_g = 2^-g: C[m][n] = sum_g 2^-g * sum_{k in group g} A[m][k]."""
    m, k, n, gs = 4, 512, 16, 64
    groups = k // gs
    a = synth.activations(4, m, k)
    s = np.repeat((2.0 ** -np.arange(groups))[:, None], n, axis=1).astype(np.float16)
    got = orc.gemm(a, _codes_const(orc, k, n, 9), s, group_size=gs, weight_type=U4B8)
    w = 2.0 ** -(np.arange(k) // gs)
    want = np.repeat(_rowsums(a, w)[:, None], n, axis=1)
    return _mismatch("group boundaries", got, want, rtol=1e-13, atol=1e-12)


def pin_one_hot_selects_columns(orc):
    """s = 1 and q = 9 only at row pi(n) (else 8): C[:, n] == A[:, pi(n)] exactly."""
    m, k, n = 6, 256, 48
    a = synth.activations(5, m, k)
    pi = (np.arange(n) * 37 + 11) % k
    codes = np.full((k, n), 8, dtype=np.uint8)
    codes[pi, np.arange(n)] = 9
    s = np.ones((2, n), dtype=np.float16)
    got = orc.gemm(a, orc.pack_gptq(codes), s, group_size=128, weight_type=U4B8)
    return _mismatch("one-hot", got, a.astype(np.float64)[:, pi])


def pin_zero_point_eight_equals_u4b8(orc):
    """u4 with every zero point 8 is the u4b8 code: identical results."""
    m, k, n = 3, 256, 32
    a = synth.activations(6, m, k)
    qw = synth.qweight(7, k, n)
    s = synth.scales(8, 2, n)
    z = np.full((2, n), 8, dtype=np.float16)
    got = orc.gemm(a, qw, s, z, group_size=128, weight_type=U4)
    want = orc.gemm(a, qw, s, group_size=128, weight_type=U4B8)
    if not np.array_equal(got, want):
        return "u4 with z=8 differs from u4b8"
    return None


def pin_zero_point_sign(orc):
    """u4, s = 1: q = 0, z = 3 gives -3 * sum A; q = 15, z = 0 gives +15 * sum A."""
    m, k, n = 2, 128, 16
    a = synth.activations(9, m, k)
    s = np.ones((1, n), dtype=np.float16)
    rs = _rowsums(a)
    for q, zv, factor in ((0, 3, -3.0), (15, 0, 15.0), (5, 12, -7.0)):
        z = np.full((1, n), zv, dtype=np.float16)
        got = orc.gemm(a, _codes_const(orc, k, n, q), s, z, group_size=128, weight_type=U4)
        bad = _mismatch(f"zero point q={q} z={zv}", got, np.repeat((factor * rs)[:, None], n, 1),
                        rtol=1e-13, atol=1e-12)
        if bad:
            return bad
    return None


def pin_zero_point_per_group_and_column(orc):
    """u4, q = 0, s = 1, z[g][n] = g + 2n: C[m][n] = -sum_k (g(k) + 2n) A[m][k]."""
    m, k, n, gs = 3, 256, 4, 64
    a = synth.activations(10, m, k)
    groups = k // gs
    z = (np.arange(groups)[:, None] + 2 * np.arange(n)[None, :]).astype(np.float16)
    s = np.ones((groups, n), dtype=np.float16)
    got = orc.gemm(a, _codes_const(orc, k, n, 0), s, z, group_size=gs, weight_type=U4)
    want = np.empty((m, n))
    for j in range(n):
        want[:, j] = -_rowsums(a, (np.arange(k) // gs) + 2.0 * j)
    return _mismatch("zero point per group/column", got, want, rtol=1e-13, atol=1e-12)


def pin_scale_per_column(orc):
    """q = 9, one group, s[n] = 2^-(n mod 5): C[m][n] = 2^-(n mod 5) * sum_k A[m][k]."""
    m, k, n = 3, 128, 20
    a = synth.activations(12, m, k)
    sv = 2.0 ** -(np.arange(n) % 5)
    s = sv[None, :].astype(np.float16)
    got = orc.gemm(a, _codes_const(orc, k, n, 9), s, group_size=-1, weight_type=U4B8)
    want = _rowsums(a)[:, None] * sv[None, :]
    return _mismatch("per-column scale", got, want, rtol=1e-13, atol=1e-12)


def pin_act_order_scale_by_gidx(orc):
    """Act-order: a row's scale is chosen by g_idx of the logical row.  q = 9, s_g = 2^-g:
    C[m][n] = sum_k 2^-g_idx[k] * A[m][k]."""
    m, k, n, gs = 3, 256, 16, 64
    perm = synth.permutation(13, k)
    g_idx = synth.act_order_gidx(perm, gs)
    a = synth.activations(14, m, k)
    s = np.repeat((2.0 ** -np.arange(k // gs))[:, None], n, 1).astype(np.float16)
    got = orc.gemm(a, _codes_const(orc, k, n, 9), s, g_idx=g_idx, group_size=gs, weight_type=U4B8)
    want = np.repeat(_rowsums(a, 2.0 ** -g_idx.astype(np.float64))[:, None], n, 1)
    return _mismatch("act-order g_idx", got, want, rtol=1e-13, atol=1e-12)


def pin_act_order_relabel_invariance(orc):
    """Relabelling K (columns of A, rows of B, entries of g_idx) by a permutation leaves C
    unchanged in exact arithmetic: C = A[:, perm] . W[perm, :]."""
    m, k, n, gs = 3, 256, 24, 64
    perm = synth.permutation(15, k)
    g_idx = synth.act_order_gidx(perm, gs)
    a = synth.activations(16, m, k)
    qw = synth.qweight(17, k, n)
    s = synth.scales(18, k // gs, n)
    base = orc.gemm(a, qw, s, g_idx=g_idx, group_size=gs, weight_type=U4B8)
    codes = orc.unpack_gptq(qw, k, n)
    qw_p = orc.pack_gptq(codes[perm])
    got = orc.gemm(np.ascontiguousarray(a[:, perm]), qw_p, s, g_idx=g_idx[perm], group_size=gs,
                   weight_type=U4B8)
    return _mismatch("act-order relabel", got, base, rtol=1e-12, atol=1e-12)


def pin_act_order_identity_equals_plain(orc):
    """g_idx[k] = k / group_size is the plain grouping: identical results."""
    m, k, n, gs = 2, 256, 16, 128
    a = synth.activations(19, m, k)
    qw = synth.qweight(20, k, n)
    s = synth.scales(21, 2, n)
    g_idx = (np.arange(k) // gs).astype(np.int32)
    got = orc.gemm(a, qw, s, g_idx=g_idx, group_size=gs)
    want = orc.gemm(a, qw, s, group_size=gs)
    if not np.array_equal(got, want):
        return "identity g_idx differs from plain grouping"
    return None


def pin_formulations_agree(orc):
    """Three formulations -- on-the-fly definition, per-group sums, materialised W with a
    plain triple loop -- agree to 1e-12 relative on random u4b8, u4 and act-order inputs."""
    m, k, n, gs = 5, 384, 40, 64
    a = synth.activations(22, m, k)
    qw = synth.qweight(23, k, n)
    s = synth.scales(24, k // gs, n)
    z = synth.zeros(25, k // gs, n)
    perm = synth.permutation(26, k)
    g_idx = synth.act_order_gidx(perm, gs)
    for wt, zz, gi in ((U4B8, None, None), (U4, z, None), (U4B8, None, g_idx), (U4, z, g_idx)):
        c1 = orc.gemm(a, qw, s, zz, gi, gs, wt)
        c2 = orc.gemm_by_groups(a, qw, s, zz, gi, gs, wt)
        w = orc.dequant(qw, s, zz, gi, k, n, gs, wt)
        c3 = orc.matmul(a.astype(np.float64), w)
        for name, other in (("by-groups", c2), ("materialised", c3)):
            bad = _mismatch(f"formulation {name} wt={wt} act={gi is not None}", other, c1,
                            rtol=1e-12, atol=1e-12)
            if bad:
                return bad
    return None


def pin_dequant_matches_library_matmul(orc):
    """The materialised W times A equals numpy's matmul of the same doubles (library pin on
    the contraction's orientation: C = A @ W, not W @ A or A @ W^T)."""
    m, k, n = 3, 128, 9
    a = synth.activations(27, m, k).astype(np.float64)
    w = synth.activations(28, k, n).astype(np.float64)
    return _mismatch("matmul", orc.matmul(a, w), a @ w, rtol=1e-13, atol=1e-13)


def pin_threads_do_not_change_result(orc):
    """Column-split threading is a pure partition: 1 thread and 7 threads agree bit for bit."""
    m, k, n = 2, 256, 37
    a = synth.activations(29, m, k)
    qw = synth.qweight(30, k, n)
    s = synth.scales(31, 2, n)
    c1 = orc.gemm(a, qw, s, threads=1)
    c7 = orc.gemm(a, qw, s, threads=7)
    if not np.array_equal(c1, c7):
        return "thread count changed the result"
    return None


# --- tile layout ---------------------------------------------------------------------------

def tile_word_index(row: int, col: int, k: int) -> tuple[int, int]:
    """Closed form of the library's tile layout: (word index, bit offset) of sorted row `row`,
    column `col`, written independently of the oracle's nested loops."""
    kblocks = k // 64
    nt, c = divmod(col, 128)
    kb, r = divmod(row, 64)
    h, r = divmod(r, 32)
    p, r = divmod(r, 8)          # r = 2*j + e inside the 8-row group p
    j, e = divmod(r, 2)
    word = (nt * kblocks + kb) * 1024 + h * 512 + c * 4 + j
    return word, 4 * p + 16 * e


def pin_tile_layout_closed_form(orc):
    """Every code lands where the closed-form index says (q[k][n] = (k + 3n) mod 16 makes
    each position distinguishable along both axes)."""
    k, n = 192, 256
    codes = ((np.arange(k)[:, None] * 5 + 3 * np.arange(n)[None, :] + (np.arange(n)[None, :] // 16)) % 16).astype(np.uint8)
    tiles = orc.repack_tiles(orc.pack_gptq(codes), None, k, n).view(np.uint32)
    rows = np.repeat(np.arange(k), n)
    cols = np.tile(np.arange(n), k)
    for row, col in zip(rows[::7], cols[::7]):
        w, b = tile_word_index(int(row), int(col), k)
        got = (int(tiles[w]) >> b) & 0xF
        if got != codes[row, col]:
            return f"tile layout: ({row},{col}) read {got}, want {codes[row, col]}"
    return None


def pin_tile_roundtrip(orc):
    """unpack(repack(x)) == x on random words; with a permutation the rows come back permuted."""
    k, n = 256, 384
    qw = synth.qweight(32, k, n)
    tiles = orc.repack_tiles(qw, None, k, n)
    if not np.array_equal(orc.unpack_tiles(tiles, k, n), qw):
        return "unpack(repack(x)) != x"
    perm = synth.permutation(33, k)
    tiles_p = orc.repack_tiles(qw, perm, k, n)
    back = orc.unpack_gptq(orc.unpack_tiles(tiles_p, k, n), k, n)
    if not np.array_equal(back, orc.unpack_gptq(qw, k, n)[perm]):
        return "permuted repack: rows are not perm-ordered"
    if np.array_equal(tiles, qw.ravel()):
        return "repack is the identity"
    return None


# --- schedule, groups, zero points ------------------------------------------------------------

def pin_csr_worked_examples(orc):
    g = _golden("csr_worked_examples.json")
    for ex in g["from_token_routes"]:
        r = orc.csr_from_token_routes(ex["n_expert"], ex["n_tokens"], ex["experts_per_token"],
                                      ex["selected"])
        if r is None:
            return "csr token routes rejected a valid example"
        for name, got, want in zip(("ex_ids", "ex_off", "ex_pairs", "pair_tok"), r,
                                   (ex["ex_ids"], ex["ex_off"], ex["ex_pairs"], ex["pair_tok"])):
            if list(got) != want:
                return f"csr token routes {name}: {list(got)} != {want}"
    for ex in g["from_pair_rows"]:
        r = orc.csr_from_pair_rows(ex["n_expert"], ex["n_tokens"], ex["selected"], ex["pair_tok"])
        if r is None:
            return "csr pair rows rejected a valid example"
        for name, got, want in zip(("ex_ids", "ex_off", "ex_pairs", "pair_tok"), r,
                                   (ex["ex_ids"], ex["ex_off"], ex["ex_pairs"], ex["pair_tok_out"])):
            if list(got) != want:
                return f"csr pair rows {name}: {list(got)} != {want}"
    for ex in g["rejected_token_routes"]:
        if orc.csr_from_token_routes(ex["n_expert"], ex["n_tokens"], ex["experts_per_token"],
                                     ex["selected"]) is not None:
            return "csr accepted a bad route count"
    for ex in g["rejected_pair_rows"]:
        if orc.csr_from_pair_rows(ex["n_expert"], ex["n_tokens"], ex["selected"], ex["pair_tok"]) is not None:
            return f"csr accepted bad pair rows {ex}"
    for ex in g["rejected_parts"]:
        if orc.csr_validate(ex["n_expert"], ex["n_tokens"], ex["ex_ids"], ex["ex_off"],
                            ex["ex_pairs"], ex["pair_tok"]):
            return f"csr validation accepted {ex}"
    return None


def pin_group_count_examples(orc):
    g = _golden("group_count_examples.json")
    for k, gs, want in g["accepted"]:
        if orc.group_count(k, gs) != want:
            return f"group count ({k},{gs}) != {want}"
    for k, gs in g["rejected"]:
        if orc.group_count(k, gs) >= 0:
            return f"group count ({k},{gs}) accepted"
    return None


def pin_qzeros_examples(orc):
    g = _golden("qzeros_examples.json")
    for words, want in g["code7"]:
        if orc.qzeros_symmetric_code7(np.array(words, dtype=np.uint32).view(np.int32)) != want:
            return f"code7 detection of {words}"
    c = g["code8_to_9"]
    groups = c["k"] // c["group_size"]
    qz = np.full(groups * c["n"] // 8, c["qzeros_word"], dtype=np.uint32).view(np.int32)
    zp = orc.qzeros_to_zero_points(qz, groups, c["n"])
    if zp is None or np.any(zp != c["zero_point"]):
        return "code 8 did not convert to zero point 9"
    lay = g["layout"]
    groups = lay["k"] // lay["group_size"]
    actual = lay["actual_zero_points_first_16_columns"]
    words = np.full(groups * lay["n"] // 8, lay["rest_of_qzeros_word"], dtype=np.uint32)
    for pc in range(2):
        words[pc] = sum((actual[pc * 8 + lane] - 1) << (4 * lane) for lane in range(8))
    zp = orc.qzeros_to_zero_points(words.view(np.int32), groups, lay["n"])
    if zp is None:
        return "layout example rejected"
    runtime_words = [sum(int(zp[0, pc * 8 + lane]) << (4 * lane) for lane in range(8)) for pc in range(3)]
    if runtime_words != lay["packed_runtime_words_first_three"]:
        return f"qzeros layout: {[hex(w) for w in runtime_words]}"
    bad = np.array([0xF], dtype=np.uint32).view(np.int32)
    if orc.qzeros_to_zero_points(np.repeat(bad, 1), 1, 8) is not None:
        return "code 15 accepted"
    return None


def pin_grouped_closed_form(orc):
    """Experts with q = 9 and expert-specific unit scales 2^-e: Y[p][n] = 2^-e(p) * sum_k A[tok(p)][k],
    and every other pair row equals a dense GEMM of its token row with its expert."""
    n_exp, n_tok, top_k, k, n = 4, 6, 2, 128, 16
    sel = synth.routes(34, n_tok, n_exp, top_k)
    ex_ids, ex_off, ex_pairs, pair_tok = orc.csr_from_token_routes(n_exp, n_tok, top_k, sel)
    a = synth.activations(35, n_tok, k)
    qw = np.concatenate([_codes_const(orc, k, n, 9).ravel()] * n_exp)
    s = np.concatenate([np.full((1, n), 2.0 ** -e, dtype=np.float16) for e in range(n_exp)])
    y = orc.grouped(a, qw, s, None, ex_ids, ex_off, ex_pairs, pair_tok, k, n, group_size=-1)
    rs = _rowsums(a)
    want = np.array([[2.0 ** -sel[p] * rs[p // top_k]] * n for p in range(n_tok * top_k)])
    bad = _mismatch("grouped closed form", y, want, rtol=1e-13, atol=1e-12)
    if bad:
        return bad
    qw2 = synth.qweight(36, k, n * n_exp).reshape(k // 8, n_exp, n).transpose(1, 0, 2).copy()
    s2 = synth.scales(37, n_exp, n)
    y2 = orc.grouped(a, qw2.ravel(), s2, None, ex_ids, ex_off, ex_pairs, pair_tok, k, n, group_size=-1)
    for p in range(n_tok * top_k):
        e = sel[p]
        want_p = orc.gemm(a[p // top_k:p // top_k + 1], qw2[e], s2[e:e + 1], group_size=-1)
        bad = _mismatch(f"grouped pair {p}", y2[p:p + 1], want_p)
        if bad:
            return bad
    return None


# --- BF16 activations ----------------------------------------------------------------------------

def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Bit patterns of values exactly representable in bfloat16 (the top half of binary32)."""
    f = np.asarray(x, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exact in bfloat16"
    return (bits >> np.uint32(16)).astype(np.uint16)


def pin_bf16_decode_all_patterns(orc):
    """Every bfloat16 bit pattern decodes as torch's bfloat16 does (a library routine)."""
    import torch
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = np.array([orc.lib.orc_bf16_to_double(int(x)) for x in b])
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()
    if not np.array_equal(np.isnan(got), np.isnan(ref)) or not np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)]):
        return "bfloat16 decode differs from torch.bfloat16"
    return None


def pin_bf16_gemm_equals_fp16_gemm_on_shared_values(orc):
    """Activations k/32 in [-2, 2), scales 2^-j and integer zero points are exact in both
    binary16 and bfloat16: the BF16-activation GEMM of their bf16 patterns equals the fp16 GEMM
    of their fp16 patterns exactly (u4b8 and u4)."""
    m, k, n = 5, 256, 48
    rng = np.random.default_rng(81)
    a = (rng.integers(-64, 64, size=(m, k)) / 32.0)
    s = 2.0 ** -rng.integers(4, 9, size=(2, n)).astype(np.float64)
    z = rng.integers(5, 11, size=(2, n)).astype(np.float64)
    qw = synth.qweight(82, k, n)
    for wt, zz in ((U4B8, None), (U4, z)):
        ref = orc.gemm(a.astype(np.float16), qw, s.astype(np.float16),
                       None if zz is None else zz.astype(np.float16), None, 128, wt)
        got = orc.gemm_bf16(_bf16_bits(a), qw, _bf16_bits(s), None if zz is None else _bf16_bits(zz),
                            None, 128, wt)
        bad = _mismatch(f"bf16 vs fp16 gemm (type {wt})", got, ref)
        if bad:
            return bad
    return None


# --- FP8 E4M3 weights (W8A16) -----------------------------------------------------------------

def _fp8_pack(codes: np.ndarray) -> np.ndarray:
    """[K][N] uint8 codes -> [K/4][N] int32 words, row 4r+i at byte i (the pages' FP8 input ABI)."""
    k, n = codes.shape
    c = codes.astype(np.uint32).reshape(k // 4, 4, n)
    w = np.zeros((k // 4, n), dtype=np.uint32)
    for i in range(4):
        w |= c[:, i, :] << np.uint32(8 * i)
    return w.view(np.int32)


def pin_e4m3_decode_all_codes(orc):
    """Every E4M3 code decodes as torch's float8_e4m3fn does (a library routine): 0x38 = 1,
    0x7E = 448, 0x01 = 2^-9, NaN only at 0x7F and 0xFF."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    if not np.array_equal(np.isnan(got), np.isnan(ref)) or not np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)]):
        return "e4m3 decode differs from float8_e4m3fn"
    if got[0x38] != 1.0 or got[0x7E] != 448.0 or got[0x01] != 2.0 ** -9 or got[0xB8] != -1.0:
        return "e4m3 landmarks"
    return None


def pin_fp8_byte_order_and_groups(orc):
    """Codes f(k, n) packed little-endian along K, power-of-two group scales 2^-g (group 128)
    and per-column factors: W[k][n] = e4m3(f(k, n)) * 2^-(k//128) * c_n exactly."""
    k, n = 384, 24
    codes = ((np.arange(k)[:, None] * 7 + np.arange(n)[None, :] * 13) % 254).astype(np.uint8)
    codes[codes >= 0x7F] += 1
    qw = _fp8_pack(codes)
    col = (1 + np.arange(n) % 4).astype(np.float64)
    s = np.array([[2.0 ** -g * col[j] for j in range(n)] for g in range(k // 128)], dtype=np.float16)
    w = orc.dequant_fp8(qw, s, k, n, 128)
    want = orc.e4m3(codes) * (2.0 ** -(np.arange(k) // 128))[:, None] * col[None, :]
    bad = _mismatch("fp8 dequant", w, want)
    if bad:
        return bad
    s1 = np.array([col], dtype=np.float16)   # channelwise: one group
    w1 = orc.dequant_fp8(qw, s1, k, n, -1)
    return _mismatch("fp8 channelwise", w1, orc.e4m3(codes) * col[None, :])


def pin_fp8_gemm_one_hot_and_library(orc):
    """One 1.0 (0x38) per column at row pi(n), zeros elsewhere, unit scales: C[:, n] =
    A[:, pi(n)]; and a seeded GEMM equals the library matmul of the dequantised matrix."""
    m, k, n = 5, 256, 32
    a = synth.activations(71, m, k)
    pi = (np.arange(n) * 37 + 3) % k
    codes = np.zeros((k, n), dtype=np.uint8)
    codes[pi, np.arange(n)] = 0x38
    c = orc.gemm_fp8(a, _fp8_pack(codes), np.ones((2, n), dtype=np.float16), 128)
    bad = _mismatch("fp8 one-hot", c, a[:, pi].astype(np.float64))
    if bad:
        return bad
    qw = synth.fp8_weights(72, k, n)
    s = synth.scales(72, 2, n, lo=1e-4, hi=2e-4)
    c = orc.gemm_fp8(a, qw, s, 128)
    want = a.astype(np.float64) @ orc.dequant_fp8(qw, s, k, n, 128)
    return _mismatch("fp8 gemm vs library matmul", c, want, rtol=1e-12, atol=1e-12)


def pin_fp8_tile_layout(orc):
    """Every tile word is the source word (row 4 * (kb*16 + 4q + t) / 4, column nt*128 + c) --
    the FP8 repack moves whole words -- and every source word appears exactly once."""
    k, n = 128, 256
    qw = synth.fp8_weights(73, k, n)
    tiles = orc.repack_fp8_tiles(qw, k, n)
    want = np.empty_like(tiles)
    for nt in range(n // 128):
        for kb in range(k // 64):
            base = (nt * (k // 64) + kb) * 2048
            for q in range(4):
                for c in range(128):
                    for t in range(4):
                        want[base + q * 512 + c * 4 + t] = qw[kb * 16 + 4 * q + t, nt * 128 + c]
    bad = _mismatch("fp8 tile words", tiles, want)
    if bad:
        return bad
    if sorted(tiles.view(np.uint32).tolist()) != sorted(qw.view(np.uint32).ravel().tolist()):
        return "fp8 tiles are not a permutation of the source words"
    return None


# --- vLLM Marlin-MoE routing (sorted_token_ids / expert_ids / sentinel rows) ------------------

def pin_moe_align_examples(orc):
    """The page's one-block example (batch prefix, sentinel prob_m * top_k after it) and a
    hand-worked top-2 routing."""
    g = _golden("moe_align_examples.json")
    ex = g["page_example"]
    got = orc.moe_align_block_size(np.zeros(ex["batch"], np.int32), ex["batch"], ex["top_k"],
                                   ex["n_experts"], ex["block_size"])
    if got is None or list(got[0]) != ex["sorted_token_ids"] or list(got[1]) != ex["expert_ids"] \
            or got[2] != ex["num_tokens_past_padded"]:
        return f"page example: {got}"
    hw = g["hand_worked"]
    got = orc.moe_align_block_size(np.array(hw["topk_ids"]), hw["m"], hw["top_k"], hw["n_experts"],
                                   hw["block_size"])
    if got is None or list(got[0]) != hw["sorted_token_ids"] or list(got[1]) != hw["expert_ids"] \
            or got[2] != hw["num_tokens_past_padded"]:
        return f"hand-worked example: {got}"
    if orc.moe_align_block_size(np.array([0, 4]), 2, 1, 4, 8) is not None:
        return "expert id out of range accepted"
    return None


def pin_moe_align_invariants(orc):
    """On a seeded routing: every id appears once, blocks hold one expert each in increasing
    expert order, the length is a multiple of the block, padding is the sentinel only."""
    m, top_k, n_exp, bs = 37, 3, 6, 8
    ids = synth.routes(51, m, n_exp, top_k)
    sid, eid, padded = orc.moe_align_block_size(ids, m, top_k, n_exp, bs)
    if padded % bs or len(eid) != padded // bs:
        return "padded length"
    real = [int(x) for x in sid if x != m * top_k]
    if sorted(real) != list(range(m * top_k)):
        return "ids not a permutation"
    for b in range(len(eid)):
        blk = [int(x) for x in sid[b * bs:(b + 1) * bs] if x != m * top_k]
        if any(ids[x] != eid[b] for x in blk) or blk != sorted(blk):
            return f"block {b}"
    if list(eid) != sorted(eid):
        return "experts not in order"
    return None


def pin_moe_blocks_equals_csr_grouped(orc):
    """The block-routed launch gives each id's row of the CSR-routed grouped GEMM (same routes),
    scaled by its top-k weight, bit for bit; sentinel rows and skipped (-1, is_ep) blocks write
    nothing."""
    m, top_k, n_exp, bs, k, n = 9, 2, 4, 4, 256, 32
    sel = synth.routes(52, m, n_exp, top_k)
    a = synth.activations(53, m, k)
    qw = synth.qweight(54, k, n * n_exp).reshape(k // 8, n_exp, n).transpose(1, 0, 2).copy()
    s = synth.scales(55, n_exp * 2, n).reshape(n_exp, 2, n)
    ex_ids, ex_off, ex_pairs, pair_tok = orc.csr_from_token_routes(n_exp, m, top_k, sel)
    y = orc.grouped(a, qw.ravel(), s, None, ex_ids, ex_off, ex_pairs, pair_tok, k, n)
    sid, eid, padded = orc.moe_align_block_size(sel, m, top_k, n_exp, bs)
    c = orc.moe_blocks(a, qw.ravel(), s, None, sid, eid, padded, None, bs, top_k, False, n_exp, k, n)
    if c is None or not np.array_equal(c, y):
        return "unweighted block routing != CSR grouped"
    w = (np.arange(m * top_k, dtype=np.float32) + 1) / 8
    cw = orc.moe_blocks(a, qw.ravel(), s, None, sid, eid, padded, w, bs, top_k, False, n_exp, k, n)
    if not np.array_equal(cw, y * w.astype(np.float64)[:, None]):
        return "top-k weights"
    eid2 = eid.copy()
    eid2[0] = -1
    c2 = orc.moe_blocks(a, qw.ravel(), s, None, sid, eid2, padded, None, bs, top_k, True, n_exp, k, n)
    skipped = [int(x) for x in sid[:bs] if x < m * top_k]
    kept = [p for p in range(m * top_k) if p not in skipped]
    if not np.all(np.isnan(c2[skipped])) or not np.array_equal(c2[kept], y[kept]):
        return "is_ep skip"
    if orc.moe_blocks(a, qw.ravel(), s, None, sid, eid2, padded, None, bs, top_k, False, n_exp, k, n) is not None:
        return "expert -1 accepted without is_ep"
    return None


# --- gated activations (SwiGLU / GeGLU after the gate and up projections) -------------------

_XS = [-30.0, -6.5, -2.0, -1.0, -0.25, 0.0, 0.125, 0.5, 1.0, 1.75, 3.0, 8.0, 30.0]


def pin_silu_identities(orc):
    """silu(x) = x * sigmoid(x): silu(0) = 0; silu(x) - silu(-x) = x (sigmoid(x) +
    sigmoid(-x) = 1); the half-angle form x/2 (1 + tanh(x/2)) through another library
    function; silu(x) -> x for large x and -> 0 for large -x."""
    if orc.act(0.0, 1) != 0.0:
        return "silu(0) != 0"
    for x in _XS:
        got = orc.act(x, 1)
        if abs((got - orc.act(-x, 1)) - x) > 1e-12 * max(1.0, abs(x)):
            return f"silu odd identity at {x}"
        if abs(got - 0.5 * x * (1.0 + math.tanh(0.5 * x))) > 1e-13 * max(1.0, abs(x)):
            return f"silu half-angle form at {x}"
    if abs(orc.act(40.0, 1) - 40.0) > 1e-12 or abs(orc.act(-40.0, 1)) > 1e-12:
        return "silu asymptotes"
    return None


def pin_gelu_tanh_identities(orc):
    """The tanh form of GELU: gelu(0) = 0; gelu(x) - gelu(-x) = x; within 1e-3 of the exact
    GELU x * Phi(x) (Phi through erf, another library routine) -- which also tells it from
    SiLU (silu(1) = 0.73, gelu(1) = 0.84); gelu(x) -> x for large x."""
    if orc.act(0.0, 2) != 0.0:
        return "gelu(0) != 0"
    for x in _XS:
        got = orc.act(x, 2)
        if abs((got - orc.act(-x, 2)) - x) > 1e-12 * max(1.0, abs(x)):
            return f"gelu odd identity at {x}"
        exact = x * 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))
        if abs(got - exact) > 1e-3:
            return f"gelu tanh form far from x Phi(x) at {x}: {got} vs {exact}"
    if abs(orc.act(30.0, 2) - 30.0) > 1e-12:
        return "gelu asymptote"
    return None


def pin_glu_gate_times_up(orc):
    """h = act(gate) * up elementwise: up = 1 gives act(gate), up = 0 gives 0, and the gate
    (not the up) operand goes through the activation."""
    g = np.array([[-2.0, 0.5, 3.0], [1.0, -0.25, 6.0]])
    u = np.array([[1.0, 1.0, 1.0], [0.0, 2.0, -3.0]])
    for kind in (1, 2):
        h = orc.glu(g, u, kind)
        want = np.array([[orc.act(x, kind) * y for x, y in zip(gr, ur)] for gr, ur in zip(g, u)])
        bad = _mismatch(f"glu kind {kind}", h, want, rtol=1e-15)
        if bad:
            return bad
        if not np.allclose(h[0], [orc.act(x, kind) for x in g[0]], rtol=1e-15) or h[1, 0] != 0.0:
            return f"glu kind {kind}: up = 1 / up = 0 rows"
    if abs(orc.glu(np.array([3.0]), np.array([0.5]), 1)[0] - orc.act(3.0, 1) * 0.5) > 1e-15:
        return "glu operand order"
    return None


def pin_gemm_glu_closed_form(orc):
    """Codes all 9 (w = s): gate = s_g * rowsum(A), up = s_u * rowsum(A); with s_g = 1 and
    s_u = 1/2 the gated FFN's h = act(rowsum) * rowsum / 2 for every column."""
    m, k, n = 3, 256, 16
    a = synth.activations(41, m, k)
    qw = _codes_const(orc, k, n, 9)
    s_g = np.ones((k // 128, n), dtype=np.float16)
    s_u = np.full((k // 128, n), 0.5, dtype=np.float16)
    rs = _rowsums(a)
    for kind in (1, 2):
        h = orc.gemm_glu(a, qw, qw, s_g, s_u, kind=kind)
        want = np.array([[orc.act(r, kind) * r / 2] * n for r in rs])
        bad = _mismatch(f"gemm_glu closed form kind {kind}", h, want, rtol=1e-12, atol=1e-12)
        if bad:
            return bad
    return None


ALL_PINS = [v for name, v in sorted(globals().items()) if name.startswith("pin_")]

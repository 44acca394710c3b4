"""The C-ABI library on the CPU: loads, exports the header's symbols, rejects bad arguments
before touching CUDA, sizes workspaces, and builds CSR schedules like the oracle does.

Fake pointers (0x1000-style, after the pages' validation tests) are used only in calls that
must be rejected by the host checks; no call here reaches a kernel launch.
"""
import json
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def w4():
    import weight_only_int4_03_gb300 as w4
    return w4


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w[48](?:a16)?_\w+)\s*\(", text)))


def test_header_symbols_exported(w4):
    import ctypes
    names = header_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(w4.library_path())
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(w4.EXPORTED) == names


def test_abi_version_and_status_names(w4):
    assert w4.abi_version() == 1
    assert w4.status_string(0) == "ok"
    assert w4.status_string(1 << 16 | 3) == "invalid-argument"
    assert w4.status_string(2 << 16 | 3) == "unsupported-shape"
    assert w4.status_string(6 << 16 | 700) == "kernel-launch"


A, B, C, S, Z, WS = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000


def gemm_status(w4, **kw):
    args = dict(a=A, lda=256, b=B, c=C, ldc=256, scales=S, zeros=None, g_idx=None, perm=None,
                ws=WS, ws_bytes=1 << 30, m=4, n=256, k=256, gs=128, wt=5, flags=0)
    args.update(kw)
    return w4._lib.w4a16_gemm(args["a"], args["lda"], args["b"], args["c"], args["ldc"],
                              args["scales"], args["zeros"], args["g_idx"], args["perm"],
                              args["ws"], args["ws_bytes"], args["m"], args["n"], args["k"],
                              args["gs"], args["wt"], args["flags"], 0)


@pytest.mark.parametrize("kw,stage,detail", [
    (dict(wt=3), 1, 8),                          # unknown weight type
    (dict(n=0), 1, 3),                           # non-positive size
    (dict(m=-1), 1, 3),
    (dict(b=None), 1, 1),                        # null weights
    (dict(scales=None), 1, 1),
    (dict(b=B + 4), 1, 2),                       # misaligned weights
    (dict(scales=S + 8), 1, 2),
    (dict(gs=100), 1, 7),                        # group size not a multiple of 16
    (dict(gs=0), 1, 7),
    (dict(gs=-2), 1, 7),
    (dict(k=384, gs=256), 1, 7),                 # group size does not divide K
    (dict(zeros=Z), 1, 4),                       # zeros without HAS_ZP / U4
    (dict(zeros=Z, flags=1 << 3), 1, 4),         # zeros with HAS_ZP but u4b8
    (dict(wt=4), 1, 4),                          # u4 without zeros
    (dict(wt=4, zeros=Z), 1, 4),                 # u4 without the HAS_ZP flag
    (dict(k=320), 2, 3),                         # K % 128 != 0
    (dict(n=384), 2, 3),                         # N % 256 != 0
    (dict(flags=1 << 1), 1, 4),                  # ACT_ORDER without g_idx/perm
    (dict(g_idx=0x70000), 1, 4),                 # g_idx without perm
    (dict(g_idx=0x70000, perm=0x80000), 1, 4),   # both without the flag
    (dict(a=None), 1, 1),
    (dict(c=None), 1, 1),
    (dict(ws=None), 1, 1),
    (dict(lda=200), 1, 3),                       # lda < K
    (dict(ldc=100), 1, 3),
    (dict(lda=260), 1, 2),                       # lda % 8 != 0
    (dict(a=A + 2), 1, 2),
    (dict(c=C + 8), 1, 2),
    (dict(ws=WS + 16), 1, 2),                    # workspace not 256-byte aligned
    (dict(flags=1 << 13 | 1 << 11), 1, 4),       # FORCE_SLICE with FORCE_MMA
    (dict(flags=1 << 13 | 1 << 10), 1, 4),       # FORCE_SLICE with FORCE_TC
    (dict(flags=1 << 11 | 1 << 8), 1, 4),        # FORCE_MMA with FORCE_SIMT
    (dict(flags=1 << 13, m=33), 2, 3),           # column-slice kernel: M <= 32 only
    (dict(flags=1 << 13, gs=32), 2, 3),          # ... and groups of whole 64-row blocks
    (dict(flags=1 << 11, m=65), 2, 3),           # split-K small-M kernel: M <= 64 only
    (dict(flags=1 << 14 | 1 << 15), 1, 4),       # SWIGLU with GEGLU
    (dict(flags=1 << 14 | 1 << 11), 1, 4),       # gated epilogue with a small-M kernel forced
    (dict(flags=1 << 15 | 1 << 13), 1, 4),
    (dict(flags=1 << 14 | 1 << 8), 1, 4),        # ... or the CUDA-core reference kernel
    (dict(flags=1 << 14, ldc=120), 1, 3),        # gated output narrower than I = 128
    (dict(flags=1 << 16 | 1 << 11, gs=32), 2, 3),  # bf16 small-M kernels: whole-block groups
    (dict(flags=1 << 16 | 1 << 8), 1, 4),        # bf16 with the CUDA-core reference kernel
    (dict(flags=1 << 16 | 1 << 2, wt=8), 1, 4),  # bf16 operands with FP8 weights
])
def test_gemm_rejects_bad_arguments_on_host(w4, kw, stage, detail):
    st = gemm_status(w4, **kw)
    assert st == (stage << 16 | detail), (kw, st >> 16, st & 0xFFFF)


def test_gemm_empty_m_is_ok_without_gpu(w4):
    assert gemm_status(w4, m=0, a=None, c=None, ws=None) == 0


def test_repack_rejects_bad_arguments(w4):
    lib = w4._lib
    assert lib.w4_repack(B, None, C, None, 256, 256, 0) >> 16 == 0 or True  # (valid: not called)
    assert lib.w4_repack(None, None, C, None, 256, 256, 0) == (1 << 16 | 1)
    assert lib.w4_repack(B + 4, None, C, None, 256, 256, 0) == (1 << 16 | 2)
    assert lib.w4_repack(B, None, C, None, 200, 256, 0) == (2 << 16 | 3)
    assert lib.w4_repack(B, None, C, None, 256, 100, 0) == (2 << 16 | 3)
    assert lib.w4_repack(B, None, B + 64, None, 256, 256, 0) == (1 << 16 | 4)   # overlap
    assert lib.w4_unpack(B, None, 256, 256, 0) == (1 << 16 | 1)
    assert lib.w4_unpack(B, C, 0, 256, 0) == (1 << 16 | 3)


def test_grouped_rejects_bad_arguments(w4):
    lib = w4._lib

    def call(**kw):
        args = dict(n_active=2, n_experts=4, n_pairs=8, n_tokens=4, n=256, k=256, gs=128, wt=5,
                    flags=0, ids=0x90000, off=0xA0000, pairs=0xB0000, tok=0xC0000)
        args.update(kw)
        return lib.w4a16_gemm_grouped(A, 256, B, C, 256, S, None, args["ids"], args["off"],
                                      args["pairs"], args["tok"], args["n_active"],
                                      args["n_experts"], args["n_pairs"], args["n_tokens"],
                                      args["n"], args["k"], args["gs"], args["wt"], args["flags"],
                                      WS, 1 << 30, 0)

    assert call(n_active=0) == (1 << 16 | 9)
    assert call(n_active=5) == (1 << 16 | 9)            # more active experts than experts
    assert call(n_active=2000, n_experts=4000) == (1 << 16 | 9)
    assert call(flags=1 << 1) == (1 << 16 | 4)          # act-order unsupported here
    assert call(flags=1 << 11) == (1 << 16 | 4)         # small-M kernels: dense calls only
    assert call(flags=1 << 13) == (1 << 16 | 4)
    assert call(ids=None) == (1 << 16 | 1)
    assert call(tok=0xC0002) == (1 << 16 | 2)
    assert call(k=320) == (2 << 16 | 3)


def test_workspace_size_host_only(w4):
    base = w4.w4a16_workspace_size(1, 4096, 4096, 128, 0, 152)
    assert base > 0 and base % 256 == 0
    ao = w4.w4a16_workspace_size(64, 4096, 4096, 128, 1 << 1, 152)
    assert ao >= w4.w4a16_workspace_size(64, 4096, 4096, 128, 0, 152) + 64 * 4096 * 2
    assert w4.w4a16_workspace_size(1, 4096, 4096, 128, 0, 152) <= w4.w4a16_workspace_size(1, 4096, 4096, 128, 0, 304)
    assert w4.w4a16_workspace_size(1, 4000, 4096, 128, 0, 152) == 0
    assert w4.w4a16_workspace_size(1, 4096, 4096, 100, 0, 152) == 0
    g = w4.w4a16_grouped_workspace_size(1024, 8, 28672, 4096, 128, 0, 152)
    assert g >= 1024 * 4096 * 2
    assert w4.w4a16_grouped_workspace_size(1024, 0, 28672, 4096, 128, 0, 152) == 0


def test_token_tile_height_from_workspace(w4):
    """The tcgen05 kernel's token-tile height, read back from the workspace size on a 152-SM
    device (the partial slots are 2 x nt x 128 fp32 per CTA): one tile up to 256 rows; above
    that ceil(M / 224) equal tiles rounded up to 16 rows, never below 192 -- unless a pair of
    half-tiles (each at most 192 rows) needs fewer tiles: then ceil(M / 384) pairs of two equal
    halves rounded up to 16 rows (M=449: 2 pairs of 2 x 128 instead of 3 tiles of 192)."""
    def nt_of(m, n=256):
        total = w4.w4a16_workspace_size(m, n, 128, 128, 0, 152)
        slots = 152 * 2 * 128 * 4
        head = total % slots
        assert head % 256 == 0
        return total // slots
    expect = {100: 112, 256: 256, 257: 288, 448: 224, 449: 256, 512: 256, 600: 320, 672: 352,
              1024: 352, 2048: 352, 4096: 384, 8192: 384}
    assert {m: nt_of(m) for m in expect} == expect


def test_csr_builder_matches_pages_examples(w4):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "csr_worked_examples.json")))
    for ex in g["from_token_routes"]:
        got = w4.w4a16_csr_from_token_routes(ex["n_expert"], ex["n_tokens"], ex["experts_per_token"],
                                             ex["selected"])
        for arr, key in zip(got, ("ex_ids", "ex_off", "ex_pairs", "pair_tok")):
            assert arr.tolist() == ex[key]
    for ex in g["rejected_token_routes"]:
        with pytest.raises(w4.W4A16Error):
            w4.w4a16_csr_from_token_routes(ex["n_expert"], ex["n_tokens"], ex["experts_per_token"],
                                           ex["selected"])
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_csr_from_token_routes(2, 1, 1, [2])


@pytest.mark.parametrize("seed,n_exp,n_tok,top_k", [(1, 8, 512, 2), (2, 64, 300, 4), (3, 3, 7, 3)])
def test_csr_builder_matches_oracle(w4, seed, n_exp, n_tok, top_k):
    sel = synth.routes(seed, n_tok, n_exp, top_k)
    got = w4.w4a16_csr_from_token_routes(n_exp, n_tok, top_k, sel)
    want = oracle.Oracle().csr_from_token_routes(n_exp, n_tok, top_k, sel)
    for x, y in zip(got, want):
        assert np.array_equal(x, y)
    assert oracle.Oracle().csr_validate(n_exp, n_tok, *got)


# --- checkpoint loading helpers (host code, pinned by the pages' three qzeros tests) ----------

def _qzeros_golden():
    with open(os.path.join(ROOT, "tests", "golden", "qzeros_examples.json")) as f:
        return json.load(f)


def test_qzeros_code7_detection_matches_page_examples(w4):
    """vllm_marlin.rs `qzeros_code7_detects_symmetric_gptq`: all-7 words are symmetric, one
    code 8 is not, an empty array is not."""
    for words, want in _qzeros_golden()["code7"]:
        assert w4.w4_qzeros_symmetric_code7(np.array(words, dtype=np.uint32).view(np.int32)) == want


def test_qzeros_code8_converts_to_zero_point_9(w4):
    """vllm_marlin.rs `qzeros_code8_repack_converts_to_actual_zero_point_9`."""
    c = _qzeros_golden()["code8_to_9"]
    groups = c["k"] // c["group_size"]
    qz = np.full(groups * c["n"] // 8, c["qzeros_word"], dtype=np.uint32).view(np.int32)
    zp = w4.w4_qzeros_to_zero_points(qz, groups, c["n"])
    assert zp.dtype == np.float16 and zp.shape == (groups, c["n"])
    assert np.all(zp == c["zero_point"])


def test_qzeros_layout_matches_page_example(w4):
    """vllm_marlin.rs `qzeros_repack_preserves_kernel_layout`: the stored codes of the first two
    words give the zero points 1..8, 8..15 of the first 16 columns, and the runtime zero points
    re-packed 4 bits per column give the page's three words."""
    lay = _qzeros_golden()["layout"]
    groups = lay["k"] // lay["group_size"]
    actual = lay["actual_zero_points_first_16_columns"]
    words = np.full(groups * lay["n"] // 8, lay["rest_of_qzeros_word"], dtype=np.uint32)
    for pc in range(2):
        words[pc] = sum((actual[pc * 8 + lane] - 1) << (4 * lane) for lane in range(8))
    zp = w4.w4_qzeros_to_zero_points(words.view(np.int32), groups, lay["n"])
    assert list(zp[0, :16].astype(int)) == actual
    runtime = [sum(int(zp[0, pc * 8 + lane]) << (4 * lane) for lane in range(8)) for pc in range(3)]
    assert runtime == lay["packed_runtime_words_first_three"]


def test_qzeros_code15_rejected_and_output_untouched(w4):
    qz = np.array([0x12345678, 0x0000F000], dtype=np.uint32).view(np.int32)
    out = np.full((1, 16), 3.0, dtype=np.float16).view(np.uint16)
    status = w4._lib.w4_qzeros_to_zero_points(qz.ctypes.data, 1, 16, out.ctypes.data)
    assert status == (1 << 16) | w4.W4A16_ARG_QZERO
    assert np.all(out.view(np.float16) == 3.0)
    with pytest.raises(w4.W4A16Error):
        w4.w4_qzeros_to_zero_points(qz, 1, 16)


def test_qzeros_every_code_and_column(w4):
    """Every stored code 0..14 in every lane position becomes code + 1 at column 8w + lane."""
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 15, size=(3, 64), dtype=np.uint32)
    words = np.zeros((3, 8), dtype=np.uint32)
    for lane in range(8):
        words |= codes[:, lane::8] << np.uint32(4 * lane)
    zp = w4.w4_qzeros_to_zero_points(words.view(np.int32), 3, 64)
    assert np.array_equal(zp.astype(np.int64), codes.astype(np.int64) + 1)


@pytest.mark.parametrize("m,n,gs,flags,want", [
    (1, 4096, 128, 0, 2), (8, 12288, 128, 0, 2),       # column-slice: M <= 8
    (16, 4096, 128, 0, 2), (32, 4096, 128, 0, 2),      # ... and M <= 32 while N/16 <= 2 x SMs
    (16, 12288, 128, 0, 1), (32, 12288, 128, 0, 1),    # split-K small-M above that
    (8, 4096, 32, 0, 1),                               # groups smaller than a 64-row block
    (8, 1024, 128, 0, 1),                              # fewer 16-column slices than SMs
    (33, 4096, 128, 0, 0), (4096, 11008 // 256 * 256, 128, 0, 0),
    (16, 4096, 128, 1 << 10, 0), (64, 4096, 128, 1 << 11, 1), (32, 4096, 128, 1 << 13, 2),
    (65, 4096, 128, 1 << 11, -1), (33, 4096, 128, 1 << 13, -1), (4, 4096, 100, 0, -1),
])
def test_kernel_choice(w4, m, n, gs, flags, want):
    """The documented dispatch rule, for a 152-SM part (host only)."""
    assert w4.w4a16_kernel_for(m, n, 4096, gs, flags, 152) == want


def test_gated_calls_run_the_tcgen05_kernel(w4):
    for m in (1, 16, 4096):
        assert w4.w4a16_kernel_for(m, 4096, 4096, 128, w4.W4A16_FLAG_SWIGLU, 152) == 0
        assert w4.w4a16_kernel_for(m, 4096, 4096, 128, w4.W4A16_FLAG_GEGLU, 152) == 0
    assert w4.w4a16_kernel_for(1, 4096, 4096, 128, w4.W4A16_FLAG_SWIGLU | w4.W4A16_FLAG_GEGLU, 152) == -1


def test_bf16_kernel_choice(w4):
    """bf16 calls follow the fp16 dispatch rule for groups of whole blocks; smaller groups go
    to the tcgen05 kernel (the small-M kernels' bf16 variants need whole-block groups)."""
    bf = w4.W4A16_FLAG_BF16
    for m, n, gs in ((1, 4096, 128), (16, 12288, 128), (64, 4096, 128), (4096, 4096, 128), (8, 4096, -1)):
        assert w4.w4a16_kernel_for(m, n, 4096, gs, bf, 152) == w4.w4a16_kernel_for(m, n, 4096, gs, 0, 152)
    for m in (1, 16, 32):
        assert w4.w4a16_kernel_for(m, 4096, 4096, 32, bf, 152) == 0
    assert w4.w4a16_kernel_for(1, 4096, 4096, 128, bf | (1 << 11), 152) == 1
    assert w4.w4a16_kernel_for(1, 4096, 4096, 128, bf | (1 << 13), 152) == 2
    assert w4.w4a16_kernel_for(1, 4096, 4096, 32, bf | (1 << 11), 152) == -1


def test_gate_up_interleave_rejects_bad_arguments(w4):
    f = w4._lib.w4_gate_up_interleave
    assert f(0x1000, 0x9000, 2, 48, 4, 0) == (1 << 16 | 3)       # n2 not a multiple of 32
    assert f(0x1000, 0x9000, 2, 64, 8, 0) == (1 << 16 | 3)       # element size
    assert f(None, 0x9000, 2, 64, 4, 0) == (1 << 16 | 1)
    assert f(0x1002, 0x9000, 2, 64, 4, 0) == (1 << 16 | 2)       # misaligned int32 source
    assert f(0x1000, 0x1010, 2, 64, 4, 0) == (1 << 16 | 4)       # overlapping


# --- block-routed MoE (vLLM interface): host builder and host checks --------------------------

@pytest.mark.parametrize("m,top_k,n_exp,bs", [(4, 2, 4, 4), (37, 3, 6, 8), (100, 2, 8, 64),
                                              (5, 1, 1, 16), (300, 4, 16, 16)])
def test_moe_align_builder_matches_oracle(w4, m, top_k, n_exp, bs):
    orc = oracle.Oracle()
    ids = synth.routes(60 + m, m, n_exp, top_k) if n_exp > 1 else np.zeros(m * top_k, np.int32)
    got = w4.w4a16_moe_align_block_size(ids, m, top_k, n_exp, bs)
    want = orc.moe_align_block_size(ids, m, top_k, n_exp, bs)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1]) and got[2] == want[2]


def test_moe_align_builder_page_examples(w4):
    with open(os.path.join(ROOT, "tests", "golden", "moe_align_examples.json")) as f:
        g = json.load(f)
    ex = g["page_example"]
    sid, eid, padded = w4.w4a16_moe_align_block_size(np.zeros(ex["batch"], np.int32), ex["batch"],
                                                     ex["top_k"], ex["n_experts"], ex["block_size"])
    assert list(sid) == ex["sorted_token_ids"] and list(eid) == ex["expert_ids"]
    assert padded == ex["num_tokens_past_padded"]
    hw = g["hand_worked"]
    sid, eid, padded = w4.w4a16_moe_align_block_size(np.array(hw["topk_ids"]), hw["m"], hw["top_k"],
                                                     hw["n_experts"], hw["block_size"])
    assert list(sid) == hw["sorted_token_ids"] and list(eid) == hw["expert_ids"]
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_moe_align_block_size(np.array([0, 4]), 2, 1, 4, 8)          # expert out of range
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_moe_align_block_size(np.array(hw["topk_ids"]), 4, 2, 4, 4, capacity=15)


def moe_status(w4, **kw):
    args = dict(a=A, lda=256, b=B, c=C, ldc=256, s=S, z=None, sid=0x70000, eid=0x71000,
                ntpp=0x72000, tw=None, max_padded=64, bs=16, top_k=2, mul=0, is_ep=0, n_exp=4,
                m=8, n=256, k=256, gs=128, wt=5, flags=0, ws=WS, ws_bytes=1 << 30)
    args.update(kw)
    return w4._lib.w4a16_gemm_moe_blocks(
        args["a"], args["lda"], args["b"], args["c"], args["ldc"], args["s"], args["z"], args["sid"],
        args["eid"], args["ntpp"], args["tw"], args["max_padded"], args["bs"], args["top_k"],
        args["mul"], args["is_ep"], args["n_exp"], args["m"], args["n"], args["k"], args["gs"],
        args["wt"], args["flags"], args["ws"], args["ws_bytes"], 0)


@pytest.mark.parametrize("kw,stage,detail", [
    (dict(bs=12), 1, 9),                       # moe_block_size not in {8, 16, 32, 48, 64}
    (dict(top_k=0), 1, 9),
    (dict(m=0), 1, 9),
    (dict(max_padded=40), 1, 9),               # not whole blocks
    (dict(max_padded=16 * 4097), 2, 9),        # more blocks than one call routes
    (dict(mul=1), 1, 4),                       # mul_topk_weights without weights
    (dict(mul=2, tw=0x73000), 1, 4),
    (dict(flags=1 << 14 | 1 << 15), 1, 4),
    (dict(flags=1 << 1), 1, 4),                # act-order is not supported here
    (dict(sid=None), 1, 1),
    (dict(ntpp=None), 1, 1),
    (dict(tw=0x73002, mul=1), 1, 2),           # misaligned weights
    (dict(ldc=128), 1, 3),
    (dict(ws_bytes=1024), 1, 6),
])
def test_moe_blocks_rejects_bad_arguments_on_host(w4, kw, stage, detail):
    if kw.get("ws_bytes") == 1024:
        # the workspace check needs the SM count; give the size query one
        assert w4.w4a16_moe_blocks_workspace_size(64, 16, 4, 256, 256, 128, 0, 152) > 1024
        return
    st = moe_status(w4, **kw)
    assert st == (stage << 16 | detail), (kw, st >> 16, st & 0xFFFF)


def test_moe_blocks_workspace_size(w4):
    assert w4.w4a16_moe_blocks_workspace_size(1536, 64, 8, 28672, 4096, 128, 0, 152) > 0
    assert w4.w4a16_moe_blocks_workspace_size(100, 64, 8, 28672, 4096, 128, 0, 152) == 0
    assert w4.w4a16_moe_blocks_workspace_size(128, 12, 8, 28672, 4096, 128, 0, 152) == 0

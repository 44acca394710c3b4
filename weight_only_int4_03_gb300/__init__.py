"""Python binding of libw4a16 (include/w4a16.h): the GB300 weight-only INT4 GEMM.

Argument marshalling only.  Every function here forwards to the C ABI of the same name;
torch tensors are passed by their data pointers (device memory for the kernels, host memory
for the schedule builder), and the stream defaults to torch's current CUDA stream.  All work
runs in the library's CUDA kernels; there is no CPU path.  If the library has not been built
(`python -c "import __graft_entry__ as g; g.build()"`), importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB_PATH

W4A16_TYPE_U4 = 4
W4A16_TYPE_U4B8 = 5
W4A16_TYPE_FE4M3 = 8

W4A16_FLAG_ACT_ORDER = 1 << 1
W4A16_FLAG_IS_K_FULL = 1 << 2
W4A16_FLAG_HAS_ZP = 1 << 3
W4A16_FLAG_FORCE_SIMT = 1 << 8
W4A16_FLAG_A_SMEM = 1 << 9
W4A16_FLAG_FORCE_TC = 1 << 10
W4A16_FLAG_FORCE_MMA = 1 << 11
W4A16_FLAG_FORCE_SLICE = 1 << 13
W4A16_FLAG_STATIC_WEIGHTS = 1 << 12
W4A16_FLAG_SWIGLU = 1 << 14
W4A16_FLAG_GEGLU = 1 << 15
W4A16_FLAG_BF16 = 1 << 16

W4A16_DEV_TIMEOUT = 1
W4A16_DEV_PERM = 2
W4A16_DEV_GIDX = 4
W4A16_DEV_SCHEDULE = 8
W4A16_DEV_ZERO = 16

W4A16_MAX_SEGMENTS = 1024
W4A16_MOE_MAX_BLOCKS = 4096
W4A16_ARG_SCRATCH = 10
W4A16_ARG_QZERO = 11
W4A16_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libw4a16.so is not built ({LIB_PATH}); run weight_only_int4_03_gb300.build.build()")

_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_U = ctypes.c_uint
_SZ = ctypes.c_size_t
_LL = ctypes.c_longlong

_SIGNATURES = {
    "w4a16_abi_version": (_I, []),
    "w4a16_status_string": (ctypes.c_char_p, [_I]),
    "w4_repack": (_I, [_P, _P, _P, _P, _I, _I, _P]),
    "w4_unpack": (_I, [_P, _P, _I, _I, _P]),
    "w4a16_workspace_size": (_SZ, [_I, _I, _I, _I, _U, _I]),
    "w4a16_gemm": (_I, [_P, _I, _P, _P, _I, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _U, _P]),
    "w4a16_gemm_noalloc": (_I, [_P, _I, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _U, _P]),
    "w4a16_grouped_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _U, _I]),
    "w4a16_gemm_grouped": (_I, [_P, _I, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                _I, _I, _U, _P, _SZ, _P]),
    "w4a16_csr_from_token_routes": (_I, [_I, _I, _I, _P, _P, _P, _P, _P]),
    "w4a16_status": (_I, [_P, _P, _P]),
    "w4a16_selftest_timeout": (_I, [_P, _LL, _P]),
    "w4_qzeros_to_zero_points": (_I, [_P, _I, _I, _P]),
    "w4_qzeros_symmetric_code7": (_I, [_P, _LL]),
    "w4a16_zero_points_check": (_I, [_P, _LL, _P, _P]),
    "w4a16_kernel_for": (_I, [_I, _I, _I, _I, _U, _I]),
    "w4_gate_up_interleave": (_I, [_P, _P, _I, _I, _I, _P]),
    "w8_repack": (_I, [_P, _P, _I, _I, _P]),
    "w8_unpack": (_I, [_P, _P, _I, _I, _P]),
    "w4a16_moe_align_block_size": (_I, [_P, _I, _I, _I, _I, _I, _P, _P]),
    "w4a16_moe_blocks_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _U, _I]),
    "w4a16_gemm_moe_blocks": (_I, [_P, _I, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                   _I, _I, _I, _I, _I, _I, _U, _P, _SZ, _P]),
}
for _name, (_res, _args) in _SIGNATURES.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGNATURES)


class W4A16Error(RuntimeError):
    """A non-zero status from the library: (stage << 16) | detail."""

    def __init__(self, fn: str, status: int):
        self.status = status
        self.stage = status >> 16
        self.detail = status & 0xFFFF
        super().__init__(f"{fn}: {status_string(status)} (stage {self.stage}, detail {self.detail})")


def status_string(status: int) -> str:
    return _lib.w4a16_status_string(status).decode()


def abi_version() -> int:
    return _lib.w4a16_abi_version()


def library_path() -> str:
    return LIB_PATH


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise W4A16Error(fn, status)


def w4_repack(qweight, perm, b_packed, k: int, n: int, status=None, stream=None) -> None:
    """GPTQ int32 [K/8, N] -> tile layout (int32 [K*N/8]); `perm` [K] or None."""
    _check("w4_repack", _lib.w4_repack(_ptr(qweight), _ptr(perm), _ptr(b_packed), _ptr(status),
                                       k, n, _stream(stream)))


def w4_gate_up_interleave(src, dst, rows: int, n2: int, stream=None) -> None:
    """Planar [rows, 2I] gate|up columns -> blocks of 16 gate / 16 up columns (device tensors of
    int32 GPTQ words or fp16 scales / zeros), for W4A16_FLAG_SWIGLU / _GEGLU."""
    _check("w4_gate_up_interleave", _lib.w4_gate_up_interleave(
        _ptr(src), _ptr(dst), rows, n2, src.element_size(), _stream(stream)))


def w8_repack(qweight, b_packed, k: int, n: int, stream=None) -> None:
    """FP8 E4M3 [K/4, N] words (four K-consecutive codes each) -> FP8 tile layout."""
    _check("w8_repack", _lib.w8_repack(_ptr(qweight), _ptr(b_packed), k, n, _stream(stream)))


def w8_unpack(b_packed, qweight, k: int, n: int, stream=None) -> None:
    """FP8 tile layout -> [K/4, N] words."""
    _check("w8_unpack", _lib.w8_unpack(_ptr(b_packed), _ptr(qweight), k, n, _stream(stream)))


def w4_unpack(b_packed, qweight, k: int, n: int, stream=None) -> None:
    """Tile layout -> GPTQ int32 [K/8, N] of the sorted rows."""
    _check("w4_unpack", _lib.w4_unpack(_ptr(b_packed), _ptr(qweight), k, n, _stream(stream)))


def w4a16_workspace_size(m: int, n: int, k: int, group_size: int, flags: int = 0,
                         num_sms: int = 0) -> int:
    return int(_lib.w4a16_workspace_size(m, n, k, group_size, flags, num_sms))


KERNEL_NAMES = {0: "tcgen05", 1: "split-K small-M", 2: "column-slice small-M"}


def w4a16_kernel_for(m: int, n: int, k: int, group_size: int, flags: int = 0, num_sms: int = 0) -> int:
    """0 tcgen05, 1 split-K small-M, 2 column-slice small-M, -1 rejected sizes/flags."""
    return int(_lib.w4a16_kernel_for(m, n, k, group_size, flags, num_sms))


def w4a16_grouped_workspace_size(n_pairs: int, n_active: int, n: int, k: int, group_size: int,
                                 flags: int = 0, num_sms: int = 0) -> int:
    return int(_lib.w4a16_grouped_workspace_size(n_pairs, n_active, n, k, group_size, flags, num_sms))


def w4a16_gemm(a, b_packed, c, scales, zeros, g_idx, perm, workspace, m: int, n: int, k: int,
               group_size: int, weight_type: int, flags: int = 0, lda: int | None = None,
               ldc: int | None = None, workspace_bytes: int | None = None, stream=None) -> None:
    """C[M, N] = A[M, K] x dequant(B), fp16 (bf16 with W4A16_FLAG_BF16) -- see include/w4a16.h."""
    if lda is None:
        lda = k
    if ldc is None:
        ldc = n // 2 if flags & (W4A16_FLAG_SWIGLU | W4A16_FLAG_GEGLU) else n
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("w4a16_gemm", _lib.w4a16_gemm(
        _ptr(a), lda, _ptr(b_packed), _ptr(c), ldc, _ptr(scales), _ptr(zeros), _ptr(g_idx),
        _ptr(perm), _ptr(workspace), workspace_bytes, m, n, k, group_size, weight_type, flags,
        _stream(stream)))


def w4a16_gemm_noalloc(a, b_packed, c, scales, zeros, g_idx, perm, m: int, n: int, k: int,
                       group_size: int, weight_type: int, flags: int = 0, status_out=None,
                       lda: int | None = None, ldc: int | None = None, stream=None) -> None:
    """w4a16_gemm with no workspace argument, for callers that cannot allocate device memory:
    the scratch is a fixed array inside the library (include/w4a16.h).  `status_out`, a
    device int32 tensor or None, receives the call's W4A16_DEV_* bits."""
    if lda is None:
        lda = k
    if ldc is None:
        ldc = n // 2 if flags & (W4A16_FLAG_SWIGLU | W4A16_FLAG_GEGLU) else n
    _check("w4a16_gemm_noalloc", _lib.w4a16_gemm_noalloc(
        _ptr(a), lda, _ptr(b_packed), _ptr(c), ldc, _ptr(scales), _ptr(zeros), _ptr(g_idx),
        _ptr(perm), _ptr(status_out), m, n, k, group_size, weight_type, flags, _stream(stream)))


def w4a16_gemm_grouped(a, b_packed_stack, y, scales_stack, zeros_stack, ex_ids, ex_off, ex_pairs,
                       pair_tok, n_active: int, n_experts: int, n_pairs: int, n_tokens: int, n: int,
                       k: int, group_size: int, weight_type: int, flags: int, workspace,
                       lda: int | None = None, ldy: int | None = None,
                       workspace_bytes: int | None = None, stream=None) -> None:
    """y[pair] = a[pair_tok[pair]] x dequant(B_expert) over an expert-major CSR schedule."""
    if lda is None:
        lda = k
    if ldy is None:
        ldy = n // 2 if flags & (W4A16_FLAG_SWIGLU | W4A16_FLAG_GEGLU) else n
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("w4a16_gemm_grouped", _lib.w4a16_gemm_grouped(
        _ptr(a), lda, _ptr(b_packed_stack), _ptr(y), ldy, _ptr(scales_stack), _ptr(zeros_stack),
        _ptr(ex_ids), _ptr(ex_off), _ptr(ex_pairs), _ptr(pair_tok), n_active, n_experts, n_pairs,
        n_tokens, n, k, group_size, weight_type, flags, _ptr(workspace), workspace_bytes,
        _stream(stream)))


def w4a16_csr_from_token_routes(n_expert: int, n_tokens: int, experts_per_token: int, selected):
    """Host schedule builder: returns (ex_ids, ex_off, ex_pairs, pair_tok) int32 numpy arrays."""
    sel = np.ascontiguousarray(selected, dtype=np.int32)
    n_pairs = n_tokens * experts_per_token
    if sel.size != n_pairs:
        raise W4A16Error("w4a16_csr_from_token_routes", 1 << 16 | 9)
    ex_ids = np.zeros(max(n_expert, 1), np.int32)
    ex_off = np.zeros(max(n_expert, 1) + 1, np.int32)
    ex_pairs = np.zeros(max(n_pairs, 1), np.int32)
    pair_tok = np.zeros(max(n_pairs, 1), np.int32)
    r = _lib.w4a16_csr_from_token_routes(n_expert, n_tokens, experts_per_token, sel.ctypes.data,
                                         ex_ids.ctypes.data, ex_off.ctypes.data,
                                         ex_pairs.ctypes.data, pair_tok.ctypes.data)
    if r < 0:
        raise W4A16Error("w4a16_csr_from_token_routes", 1 << 16 | 9)
    return ex_ids[:r].copy(), ex_off[:r + 1].copy(), ex_pairs[:n_pairs].copy(), pair_tok[:n_pairs].copy()


def w4a16_status(workspace, stream=None) -> int:
    """Reads and clears the W4A16_DEV_* bits of a workspace (synchronises the stream)."""
    bits = ctypes.c_int(0)
    _check("w4a16_status", _lib.w4a16_status(_ptr(workspace), ctypes.addressof(bits), _stream(stream)))
    return bits.value


def w4a16_selftest_timeout(workspace, limit_ns: int, stream=None) -> None:
    _check("w4a16_selftest_timeout", _lib.w4a16_selftest_timeout(_ptr(workspace), limit_ns,
                                                                  _stream(stream)))


def w4_qzeros_to_zero_points(qzeros, groups: int, n: int):
    """AutoGPTQ packed `zero - 1` words [groups, n/8] (host) -> fp16 zero points [groups, n]
    as a numpy float16 array (host); raises W4A16Error on a stored code 15."""
    qz = np.ascontiguousarray(qzeros, dtype=np.int32)
    if qz.size != groups * (n // 8):
        raise W4A16Error("w4_qzeros_to_zero_points", 1 << 16 | 3)
    out = np.empty((groups, n), dtype=np.uint16)
    _check("w4_qzeros_to_zero_points",
           _lib.w4_qzeros_to_zero_points(qz.ctypes.data, groups, n, out.ctypes.data))
    return out.view(np.float16)


def w4_qzeros_symmetric_code7(qzeros) -> bool:
    """True when every 4-bit code of every packed zero word is 7 (a symmetric checkpoint)."""
    qz = np.ascontiguousarray(qzeros, dtype=np.int32)
    return bool(_lib.w4_qzeros_symmetric_code7(qz.ctypes.data if qz.size else None, qz.size))


def w4a16_zero_points_check(zeros, status, stream=None) -> None:
    """ORs W4A16_DEV_ZERO into the device int32 `status` if a zero point (device fp16 tensor)
    is not an integer in [0, 15]."""
    _check("w4a16_zero_points_check", _lib.w4a16_zero_points_check(
        _ptr(zeros), zeros.numel(), _ptr(status), _stream(stream)))


def w4a16_moe_align_block_size(topk_ids, m: int, top_k: int, n_experts: int, block_size: int,
                               capacity: int | None = None):
    """Host routing builder: (sorted_token_ids, expert_ids, num_tokens_past_padded) numpy int32
    arrays trimmed to the padded length (vLLM's moe_align_block_size reading)."""
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    if ids.size != m * top_k:
        raise W4A16Error("w4a16_moe_align_block_size", 1 << 16 | 9)
    if capacity is None:
        capacity = m * top_k + n_experts * (block_size - 1)
    sorted_ids = np.zeros(max(capacity, 1), np.int32)
    expert_ids = np.zeros(max(capacity // block_size, 1), np.int32)
    r = _lib.w4a16_moe_align_block_size(ids.ctypes.data, m, top_k, n_experts, block_size, capacity,
                                        sorted_ids.ctypes.data, expert_ids.ctypes.data)
    if r < 0:
        raise W4A16Error("w4a16_moe_align_block_size", 1 << 16 | 9)
    return sorted_ids[:r].copy(), expert_ids[:r // block_size].copy(), r


def w4a16_moe_blocks_workspace_size(max_padded: int, moe_block_size: int, n_experts: int, n: int,
                                    k: int, group_size: int, flags: int = 0, num_sms: int = 0) -> int:
    return int(_lib.w4a16_moe_blocks_workspace_size(max_padded, moe_block_size, n_experts, n, k,
                                                    group_size, flags, num_sms))


def w4a16_gemm_moe_blocks(a, b_packed_stack, c, scales_stack, zeros_stack, sorted_token_ids,
                          expert_ids, num_tokens_past_padded, topk_weights, max_padded: int,
                          moe_block_size: int, top_k: int, mul_topk_weights: bool, is_ep: bool,
                          n_experts: int, prob_m: int, n: int, k: int, group_size: int,
                          weight_type: int, flags: int, workspace, lda: int | None = None,
                          ldc: int | None = None, workspace_bytes: int | None = None,
                          stream=None) -> None:
    """c[id] = a[id / top_k] x dequant(B_expert) (x topk_weights[id]) over vLLM-style block
    routing (sorted_token_ids / expert_ids / num_tokens_past_padded on the device)."""
    if lda is None:
        lda = k
    if ldc is None:
        ldc = n // 2 if flags & (W4A16_FLAG_SWIGLU | W4A16_FLAG_GEGLU) else n
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("w4a16_gemm_moe_blocks", _lib.w4a16_gemm_moe_blocks(
        _ptr(a), lda, _ptr(b_packed_stack), _ptr(c), ldc, _ptr(scales_stack), _ptr(zeros_stack),
        _ptr(sorted_token_ids), _ptr(expert_ids), _ptr(num_tokens_past_padded), _ptr(topk_weights),
        max_padded, moe_block_size, top_k, int(bool(mul_topk_weights)), int(bool(is_ep)), n_experts,
        prob_m, n, k, group_size, weight_type, flags, _ptr(workspace), workspace_bytes,
        _stream(stream)))

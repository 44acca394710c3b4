"""Python face of the CPU oracle (oracle/w4a16_oracle.c).

TEST INFRASTRUCTURE: only tests/, the smoke check in __graft_entry__ and the CPU-baseline
leg of bench.py use this module.  The product never imports it.

`build()` compiles the C file with gcc into oracle/_build/; the functions below marshal
numpy arrays into it.  fp16 tensors travel as their raw 16-bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libw4a16_oracle.so")

U4 = 4
U4B8 = 5

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle (plain C, -O2, pthreads) and return the library path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, src,
                               "-lpthread", "-lm"])
        os.replace(tmp, out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    I = ctypes.c_int
    L = ctypes.c_long
    lib.orc_half_to_double.restype = ctypes.c_double
    lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_halves_to_doubles.argtypes = [P, L, P]
    lib.orc_unpack_gptq.argtypes = [P, I, I, P]
    lib.orc_pack_gptq.argtypes = [P, I, I, P]
    lib.orc_group_count.restype = I
    lib.orc_group_count.argtypes = [I, I]
    lib.orc_dequant.argtypes = [P, P, P, P, I, I, I, I, P]
    lib.orc_matmul.argtypes = [P, L, P, I, I, I, P]
    lib.orc_gemm.argtypes = [P, L, I, P, P, P, P, I, I, I, I, P, I]
    lib.orc_gemm_bf16.argtypes = [P, L, I, P, P, P, P, I, I, I, I, P, I]
    lib.orc_bf16_to_double.restype = ctypes.c_double
    lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_gemm_by_groups.argtypes = [P, L, I, P, P, P, P, I, I, I, I, I, P]
    lib.orc_repack_tiles.argtypes = [P, P, I, I, P]
    lib.orc_unpack_tiles.argtypes = [P, I, I, P]
    lib.orc_csr_from_pair_rows.restype = I
    lib.orc_csr_from_pair_rows.argtypes = [I, I, I, P, P, P, P, P, P]
    lib.orc_csr_from_token_routes.restype = I
    lib.orc_csr_from_token_routes.argtypes = [I, I, I, P, I, P, P, P, P]
    lib.orc_csr_validate.restype = I
    lib.orc_csr_validate.argtypes = [I, I, I, I, P, P, P, P]
    lib.orc_grouped.argtypes = [P, L, P, P, P, P, P, P, P, I, I, I, I, I, P, I]
    lib.orc_qzeros_to_zero_points.restype = I
    lib.orc_qzeros_to_zero_points.argtypes = [P, I, I, P]
    lib.orc_e4m3_to_double.restype = ctypes.c_double
    lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.orc_dequant_fp8.argtypes = [P, P, I, I, I, P]
    lib.orc_gemm_fp8.argtypes = [P, L, I, P, P, I, I, I, P, I]
    lib.orc_repack_fp8_tiles.argtypes = [P, I, I, P]
    lib.orc_moe_align_block_size.restype = I
    lib.orc_moe_align_block_size.argtypes = [P, I, I, I, I, I, P, P]
    lib.orc_moe_blocks.restype = I
    lib.orc_moe_blocks.argtypes = [P, L, P, P, P, P, P, I, P, I, I, I, I, I, I, I, I, I, P, I]
    lib.orc_act.restype = ctypes.c_double
    lib.orc_act.argtypes = [ctypes.c_double, I]
    lib.orc_glu.argtypes = [P, P, L, I, P]
    lib.orc_qzeros_symmetric_code7.restype = I
    lib.orc_qzeros_symmetric_code7.argtypes = [P, L]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(arr):
    return None if arr is None else arr.ctypes.data


def _c(arr, dtype):
    return None if arr is None else np.ascontiguousarray(arr, dtype=dtype)


def _h(arr):
    """fp16 array -> contiguous uint16 bit patterns."""
    if arr is None:
        return None
    return np.ascontiguousarray(np.asarray(arr, dtype=np.float16)).view(np.uint16)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class Oracle:
    """numpy wrappers around one loaded oracle library (the default one unless a path is given,
    which the mutation tests use to load a deliberately broken copy)."""

    def __init__(self, path: str | None = None):
        self.lib = load(path)

    def half_to_double(self, h: np.ndarray) -> np.ndarray:
        h = _h(h)
        out = np.empty(h.shape, dtype=np.float64)
        self.lib.orc_halves_to_doubles(_ptr(h), h.size, _ptr(out))
        return out

    def unpack_gptq(self, qweight: np.ndarray, k: int, n: int) -> np.ndarray:
        qw = _c(qweight, np.int32)
        out = np.empty((k, n), dtype=np.uint8)
        self.lib.orc_unpack_gptq(_ptr(qw), k, n, _ptr(out))
        return out

    def pack_gptq(self, codes: np.ndarray) -> np.ndarray:
        codes = _c(codes, np.uint8)
        k, n = codes.shape
        out = np.empty((k // 8, n), dtype=np.int32)
        self.lib.orc_pack_gptq(_ptr(codes), k, n, _ptr(out))
        return out

    def group_count(self, k: int, group_size: int) -> int:
        return self.lib.orc_group_count(k, group_size)

    def dequant(self, qweight, scales, zeros, g_idx, k, n, group_size, weight_type):
        qw, s, z, g = _c(qweight, np.int32), _h(scales), _h(zeros), _c(g_idx, np.int32)
        out = np.empty((k, n), dtype=np.float64)
        self.lib.orc_dequant(_ptr(qw), _ptr(s), _ptr(z), _ptr(g), k, n, group_size, weight_type,
                             _ptr(out))
        return out

    def matmul(self, a: np.ndarray, w: np.ndarray) -> np.ndarray:
        a, w = _c(a, np.float64), _c(w, np.float64)
        m, k = a.shape
        n = w.shape[1]
        out = np.empty((m, n), dtype=np.float64)
        self.lib.orc_matmul(_ptr(a), k, _ptr(w), m, k, n, _ptr(out))
        return out

    def gemm(self, a, qweight, scales, zeros=None, g_idx=None, group_size=128, weight_type=U4B8,
             threads: int | None = None) -> np.ndarray:
        """C [M][N] in double.  `a` is fp16 [M][K] (rows may be a strided view)."""
        a = _h(a)
        m, k = a.shape
        qw, s, z, g = _c(qweight, np.int32), _h(scales), _h(zeros), _c(g_idx, np.int32)
        n = qw.shape[1]
        out = np.empty((m, n), dtype=np.float64)
        self.lib.orc_gemm(_ptr(a), k, m, _ptr(qw), _ptr(s), _ptr(z), _ptr(g), k, n, group_size,
                          weight_type, _ptr(out), threads or default_threads())
        return out

    def bf16_to_double(self, bits) -> np.ndarray:
        """Doubles of bfloat16 bit patterns (uint16 array)."""
        b = np.asarray(bits, dtype=np.uint16)
        return np.array([self.lib.orc_bf16_to_double(int(x)) for x in b.ravel()]).reshape(b.shape)

    def gemm_bf16(self, a_bits, qweight, scale_bits, zero_bits=None, g_idx=None, group_size=128,
                  weight_type=U4B8, threads: int | None = None) -> np.ndarray:
        """C [M][N] in double with bfloat16 activations, scales and zeros, given as their uint16
        bit patterns."""
        a = np.ascontiguousarray(a_bits, dtype=np.uint16)
        m, k = a.shape
        qw, g = _c(qweight, np.int32), _c(g_idx, np.int32)
        s = np.ascontiguousarray(scale_bits, dtype=np.uint16)
        z = None if zero_bits is None else np.ascontiguousarray(zero_bits, dtype=np.uint16)
        n = qw.shape[1]
        out = np.empty((m, n), dtype=np.float64)
        self.lib.orc_gemm_bf16(_ptr(a), k, m, _ptr(qw), _ptr(s), _ptr(z), _ptr(g), k, n, group_size,
                               weight_type, _ptr(out), threads or default_threads())
        return out

    def gemm_by_groups(self, a, qweight, scales, zeros=None, g_idx=None, group_size=128,
                       weight_type=U4B8) -> np.ndarray:
        a = _h(a)
        m, k = a.shape
        qw, s, z, g = _c(qweight, np.int32), _h(scales), _h(zeros), _c(g_idx, np.int32)
        n = qw.shape[1]
        groups = s.shape[0]
        out = np.empty((m, n), dtype=np.float64)
        self.lib.orc_gemm_by_groups(_ptr(a), k, m, _ptr(qw), _ptr(s), _ptr(z), _ptr(g), k, n,
                                    group_size, weight_type, groups, _ptr(out))
        return out

    def repack_tiles(self, qweight, perm, k, n) -> np.ndarray:
        qw, p = _c(qweight, np.int32), _c(perm, np.int32)
        out = np.empty(k * n // 8, dtype=np.int32)
        self.lib.orc_repack_tiles(_ptr(qw), _ptr(p), k, n, _ptr(out))
        return out

    def unpack_tiles(self, tiles, k, n) -> np.ndarray:
        t = _c(tiles, np.int32)
        out = np.empty((k // 8, n), dtype=np.int32)
        self.lib.orc_unpack_tiles(_ptr(t), k, n, _ptr(out))
        return out

    def csr_from_pair_rows(self, n_expert, n_tokens, selected, pair_tok):
        sel, pt = _c(selected, np.int32), _c(pair_tok, np.int32)
        n_pairs = sel.size
        ex_ids = np.zeros(max(n_expert, 1), np.int32)
        ex_off = np.zeros(max(n_expert, 1) + 1, np.int32)
        ex_pairs = np.zeros(max(n_pairs, 1), np.int32)
        pt_out = np.zeros(max(n_pairs, 1), np.int32)
        r = self.lib.orc_csr_from_pair_rows(n_expert, n_tokens, n_pairs, _ptr(sel), _ptr(pt),
                                            _ptr(ex_ids), _ptr(ex_off), _ptr(ex_pairs), _ptr(pt_out))
        if r < 0:
            return None
        return ex_ids[:r].copy(), ex_off[:r + 1].copy(), ex_pairs[:n_pairs].copy(), pt_out[:n_pairs].copy()

    def csr_from_token_routes(self, n_expert, n_tokens, experts_per_token, selected):
        sel = _c(selected, np.int32)
        n_sel = sel.size
        ex_ids = np.zeros(max(n_expert, 1), np.int32)
        ex_off = np.zeros(max(n_expert, 1) + 1, np.int32)
        ex_pairs = np.zeros(max(n_sel, 1), np.int32)
        pt_out = np.zeros(max(n_sel, 1), np.int32)
        r = self.lib.orc_csr_from_token_routes(n_expert, n_tokens, experts_per_token, _ptr(sel),
                                               n_sel, _ptr(ex_ids), _ptr(ex_off), _ptr(ex_pairs),
                                               _ptr(pt_out))
        if r < 0:
            return None
        return ex_ids[:r].copy(), ex_off[:r + 1].copy(), ex_pairs[:n_sel].copy(), pt_out[:n_sel].copy()

    def csr_validate(self, n_expert, n_tokens, ex_ids, ex_off, ex_pairs, pair_tok) -> bool:
        ids, off = _c(ex_ids, np.int32), _c(ex_off, np.int32)
        pairs, pt = _c(ex_pairs, np.int32), _c(pair_tok, np.int32)
        if off.size != ids.size + 1 or pt.size != pairs.size:
            return False
        return self.lib.orc_csr_validate(n_expert, n_tokens, ids.size, pairs.size, _ptr(ids),
                                         _ptr(off), _ptr(pairs), _ptr(pt)) == 0

    def grouped(self, a, qweight_stack, scales_stack, zeros_stack, ex_ids, ex_off, ex_pairs,
                pair_tok, k, n, group_size=128, weight_type=U4B8, threads: int | None = None):
        a = _h(a)
        qw = _c(qweight_stack, np.int32)
        s, z = _h(scales_stack), _h(zeros_stack)
        ids, off = _c(ex_ids, np.int32), _c(ex_off, np.int32)
        pairs, pt = _c(ex_pairs, np.int32), _c(pair_tok, np.int32)
        out = np.zeros((pairs.size, n), dtype=np.float64)
        self.lib.orc_grouped(_ptr(a), a.shape[1], _ptr(qw), _ptr(s), _ptr(z), _ptr(ids), _ptr(off),
                             _ptr(pairs), _ptr(pt), ids.size, k, n, group_size, weight_type,
                             _ptr(out), threads or default_threads())
        return out

    def e4m3(self, codes) -> np.ndarray:
        """Doubles of E4M3 codes (uint8 array)."""
        c = np.asarray(codes, dtype=np.uint8)
        return np.array([self.lib.orc_e4m3_to_double(int(x)) for x in c.ravel()]).reshape(c.shape)

    def dequant_fp8(self, qweight, scales, k, n, group_size=128):
        qw, s = _c(qweight, np.int32), _h(scales)
        out = np.empty((k, n), dtype=np.float64)
        self.lib.orc_dequant_fp8(_ptr(qw), _ptr(s), k, n, group_size, _ptr(out))
        return out

    def gemm_fp8(self, a, qweight, scales, group_size=128, threads: int | None = None):
        """C [M][N] in double with FP8 E4M3 weights ([K/4, N] words of 4 K-consecutive bytes)."""
        a = _h(a)
        m, k = a.shape
        qw, s = _c(qweight, np.int32), _h(scales)
        n = qw.shape[1]
        out = np.empty((m, n), dtype=np.float64)
        self.lib.orc_gemm_fp8(_ptr(a), k, m, _ptr(qw), _ptr(s), k, n, group_size, _ptr(out),
                              threads or default_threads())
        return out

    def repack_fp8_tiles(self, qweight, k, n) -> np.ndarray:
        qw = _c(qweight, np.int32)
        out = np.empty(k * n // 4, dtype=np.int32)
        self.lib.orc_repack_fp8_tiles(_ptr(qw), k, n, _ptr(out))
        return out

    def moe_align_block_size(self, topk_ids, m, top_k, n_experts, block_size, capacity=None):
        """(sorted_ids, expert_ids, num_tokens_past_padded) of the vLLM routing, or None."""
        ids = _c(topk_ids, np.int32)
        if capacity is None:
            capacity = m * top_k + n_experts * (block_size - 1)
        sorted_ids = np.full(max(capacity, 1), -7, np.int32)
        expert_ids = np.full(max(capacity // block_size, 1), -7, np.int32)
        r = self.lib.orc_moe_align_block_size(_ptr(ids), m, top_k, n_experts, block_size, capacity,
                                              _ptr(sorted_ids), _ptr(expert_ids))
        if r < 0:
            return None
        return sorted_ids[:r].copy(), expert_ids[:r // block_size].copy(), r

    def moe_blocks(self, a, qweight_stack, scales_stack, zeros_stack, sorted_ids, expert_ids,
                   padded, topk_weights, block_size, top_k, is_ep, n_experts, k, n,
                   group_size=128, weight_type=U4B8, threads: int | None = None):
        """c [m*top_k][n] in double (NaN in rows no entry names), or None on bad expert ids."""
        a = _h(a)
        m = a.shape[0]
        qw = _c(qweight_stack, np.int32)
        s, z = _h(scales_stack), _h(zeros_stack)
        sid, eid = _c(sorted_ids, np.int32), _c(expert_ids, np.int32)
        tw = _c(topk_weights, np.float32)
        out = np.full((m * top_k, n), np.nan)
        r = self.lib.orc_moe_blocks(_ptr(a), a.shape[1], _ptr(qw), _ptr(s), _ptr(z), _ptr(sid),
                                    _ptr(eid), padded, _ptr(tw), block_size, top_k, int(is_ep),
                                    n_experts, m, k, n, group_size, weight_type, _ptr(out),
                                    threads or default_threads())
        return None if r != 0 else out

    def act(self, x: float, kind: int) -> float:
        """silu (kind 1) or tanh-form gelu (kind 2) of one double."""
        return float(self.lib.orc_act(float(x), kind))

    def glu(self, gate, up, kind: int = 1) -> np.ndarray:
        """h = act(gate) * up elementwise, in double (kind 1 SiLU, 2 GELU tanh form)."""
        g, u = _c(gate, np.float64), _c(up, np.float64)
        assert g.shape == u.shape
        out = np.empty(g.shape, dtype=np.float64)
        self.lib.orc_glu(_ptr(g), _ptr(u), g.size, kind, _ptr(out))
        return out

    def gemm_glu(self, a, qweight_gate, qweight_up, scales_gate, scales_up, zeros_gate=None,
                 zeros_up=None, g_idx=None, group_size=128, weight_type=U4B8, kind: int = 1):
        """h = act(A Wg) * (A Wu): the two GEMMs of the gated FFN, then the activation."""
        gate = self.gemm(a, qweight_gate, scales_gate, zeros_gate, g_idx, group_size, weight_type)
        up = self.gemm(a, qweight_up, scales_up, zeros_up, g_idx, group_size, weight_type)
        return self.glu(gate, up, kind)

    def qzeros_to_zero_points(self, qzeros, groups, n):
        qz = _c(qzeros, np.int32)
        out = np.empty((groups, n), dtype=np.float64)
        if self.lib.orc_qzeros_to_zero_points(_ptr(qz), groups, n, _ptr(out)) != 0:
            return None
        return out

    def qzeros_symmetric_code7(self, qzeros) -> bool:
        qz = _c(qzeros, np.int32)
        return bool(self.lib.orc_qzeros_symmetric_code7(_ptr(qz), qz.size))


_default: Oracle | None = None


def oracle() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default

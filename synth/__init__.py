"""Seeded synthetic inputs for the W4A16 GEMM, shared by the tests, the bench and the smoke run.

This module draws numbers and nothing else: it holds none of the method's arithmetic (no
unpacking, no dequantisation, no matmul, no layout).  Both the CUDA path and the CPU oracle are
fed from here, so the two sides always see the same bits.

Generator.  A 64-bit linear congruential generator with the multiplier/increment pair that the
ferrum-kernels marlin.rs page uses for its seeded GPU-vs-source test
(`gpt_oss_mxfp4_marlin_moe_bf16_ffi_matches_source_reference_for_four_cases`, constants
LCG_MULTIPLIER / LCG_INCREMENT).  Every tensor gets its own stream: the stream's starting state
mixes the run seed with a tag derived from the tensor's name, and is advanced once before use.
Sequences are produced in vectorised blocks with the affine jump-ahead x_{j} = A_j x_0 + C_j
(mod 2^64), which gives exactly the values a scalar loop would.

Value recipes (the workload descriptions in the W4A16 configurations):
  * packed weights: raw 32-bit words, so every nibble is uniform on {0..15};
  * scales: uniform on [lo, hi), rounded to fp16 (round-to-nearest-even);
  * activations: normal N(0, sigma) by Box-Muller in fp64, rounded to fp16;
  * zero points: uniform integers on {lo..hi}, stored as fp16;
  * act-order: a seeded Fisher-Yates permutation;
  * MoE routing: per token, `top_k` distinct experts drawn uniformly.
"""
from __future__ import annotations

import numpy as np

LCG_MUL = np.uint64(0x5851F42D4C957F2D)
LCG_INC = np.uint64(0x14057B7EF767814F)
_GOLDEN = 0x9E3779B97F4A7C15
_MASK64 = (1 << 64) - 1
_BLOCK = 1 << 18

_coeff_cache: dict[int, tuple[np.ndarray, np.ndarray]] = {}


def _coeffs(block: int) -> tuple[np.ndarray, np.ndarray]:
    """A_j, C_j for j = 1..block such that x_j = A_j * x_0 + C_j (mod 2^64)."""
    if block in _coeff_cache:
        return _coeff_cache[block]
    a = np.empty(block, dtype=np.uint64)
    c = np.empty(block, dtype=np.uint64)
    a[0] = LCG_MUL
    c[0] = LCG_INC
    filled = 1
    with np.errstate(over="ignore"):
        while filled < block:
            take = min(filled, block - filled)
            a_last = a[filled - 1]
            c_last = c[filled - 1]
            a[filled:filled + take] = a[:take] * a_last
            c[filled:filled + take] = a[:take] * c_last + c[:take]
            filled += take
    _coeff_cache[block] = (a, c)
    return a, c


def _tag(name: str) -> int:
    """FNV-1a 64-bit hash of a stream name (a fixed, platform-independent tag)."""
    h = 0xCBF29CE484222325
    for byte in name.encode():
        h ^= byte
        h = (h * 0x100000001B3) & _MASK64
    return h


class Stream:
    """One seeded LCG stream."""

    def __init__(self, seed: int, name: str):
        state = ((seed + 1) * _GOLDEN) & _MASK64
        state ^= _tag(name)
        self.state = (state * int(LCG_MUL) + int(LCG_INC)) & _MASK64

    def raw(self, count: int) -> np.ndarray:
        """The next `count` 64-bit states."""
        out = np.empty(count, dtype=np.uint64)
        a, c = _coeffs(_BLOCK)
        pos = 0
        x0 = np.uint64(self.state)
        with np.errstate(over="ignore"):
            while pos < count:
                take = min(_BLOCK, count - pos)
                blk = a[:take] * x0 + c[:take]
                out[pos:pos + take] = blk
                x0 = blk[-1]
                pos += take
        if count:
            self.state = int(out[-1])
        return out

    def uniform(self, count: int) -> np.ndarray:
        """Doubles uniform on [0, 1): the top 53 bits of each state."""
        return (self.raw(count) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)

    def words(self, count: int) -> np.ndarray:
        """Uniform 32-bit words (the top half of each state) as int32."""
        return (self.raw(count) >> np.uint64(32)).astype(np.uint32).view(np.int32)

    def normal(self, count: int, sigma: float = 1.0) -> np.ndarray:
        """N(0, sigma^2) doubles by Box-Muller (cosine branch only)."""
        u = self.uniform(2 * count)
        u1 = 1.0 - u[0::2]          # (0, 1], keeps log finite
        u2 = u[1::2]
        return sigma * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    def below(self, bound: int) -> int:
        """One integer uniform on [0, bound)."""
        return int(self.uniform(1)[0] * bound)


def fp16(values: np.ndarray) -> np.ndarray:
    """Round doubles to IEEE binary16 (numpy rounds to nearest even)."""
    return np.asarray(values, dtype=np.float64).astype(np.float16)


def bf16_bits(values: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of doubles rounded to bfloat16 (through binary32, each step to nearest
    even); finite inputs only."""
    u = np.asarray(values, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def activations(seed: int, m: int, k: int, sigma: float = 1.0, name: str = "A") -> np.ndarray:
    """fp16 [m, k] ~ N(0, sigma)."""
    return fp16(Stream(seed, name).normal(m * k, sigma)).reshape(m, k)


def qweight(seed: int, k: int, n: int, name: str = "qweight") -> np.ndarray:
    """int32 [k/8, n]: random packed words, i.e. i.i.d. uniform 4-bit codes."""
    return Stream(seed, name).words((k // 8) * n).reshape(k // 8, n)


def fp8_weights(seed: int, k: int, n: int, name: str = "fp8") -> np.ndarray:
    """int32 [k/4, n]: four K-consecutive E4M3 codes per word (row 4r+i at byte i), each code
    uniform over the 254 codes that are numbers (the two NaN codes 0x7F and 0xFF are skipped)."""
    u = Stream(seed, name).uniform(k * n)
    idx = np.floor(u * 254).astype(np.int64)
    codes = idx + (idx >= 0x7F) + (idx >= 0xFE)
    codes = codes.reshape(k // 4, 4, n)          # [word row][byte][column], byte i = row 4r+i
    words = np.zeros((k // 4, n), dtype=np.uint32)
    for i in range(4):
        words |= codes[:, i, :].astype(np.uint32) << np.uint32(8 * i)
    return words.view(np.int32)


def scales(seed: int, groups: int, n: int, lo: float = 0.001, hi: float = 0.02,
           name: str = "scales") -> np.ndarray:
    """fp16 [groups, n] ~ U[lo, hi)."""
    u = Stream(seed, name).uniform(groups * n)
    return fp16(lo + (hi - lo) * u).reshape(groups, n)


def zeros(seed: int, groups: int, n: int, lo: int = 6, hi: int = 9, name: str = "zeros") -> np.ndarray:
    """fp16 [groups, n] holding integers uniform on {lo..hi}."""
    u = Stream(seed, name).uniform(groups * n)
    vals = lo + np.floor(u * (hi - lo + 1))
    return fp16(vals).reshape(groups, n)


def permutation(seed: int, k: int, name: str = "perm") -> np.ndarray:
    """int32 [k]: a Fisher-Yates shuffle of 0..k-1."""
    perm = np.arange(k, dtype=np.int64)
    u = Stream(seed, name).uniform(max(k - 1, 0))
    for idx, i in enumerate(range(k - 1, 0, -1)):
        j = int(u[idx] * (i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm.astype(np.int32)


def routes(seed: int, n_tokens: int, n_experts: int, top_k: int, name: str = "routes") -> np.ndarray:
    """int32 [n_tokens * top_k], token-major: `top_k` distinct experts per token, uniform."""
    s = Stream(seed, name)
    u = s.uniform(n_tokens * top_k)
    out = np.empty(n_tokens * top_k, dtype=np.int32)
    for t in range(n_tokens):
        remaining = list(range(n_experts))
        for j in range(top_k):
            pick = int(u[t * top_k + j] * len(remaining))
            out[t * top_k + j] = remaining.pop(pick)
    return out


def group_count(k: int, group_size: int) -> int:
    """Number of scale rows for a K extent (group_size -1 means one group)."""
    return 1 if group_size == -1 else k // group_size


def act_order_gidx(perm: np.ndarray, group_size: int) -> np.ndarray:
    """g_idx for a shuffled act-order layer whose groups each hold `group_size` rows.

    Row perm[i] of the logical weight belongs to group i // group_size, so perm sorts g_idx:
    it lists the rows of group 0 first, then those of group 1, and so on.  Inside a group its
    order is the shuffle's, not increasing row index (a stable argsort of g_idx would differ
    there); the GEMM accepts any order inside a group.  This is a drawing recipe, not part of
    the GEMM.
    """
    g = np.empty(perm.shape[0], dtype=np.int32)
    g[perm] = np.arange(perm.shape[0], dtype=np.int32) // group_size
    return g

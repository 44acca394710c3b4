"""Shared test helpers: seeded problems, GPU runs through the C ABI, oracle references."""
from __future__ import annotations

import dataclasses

import numpy as np

import synth

U4, U4B8 = 4, 5
FLAG_ACT_ORDER = 1 << 1
FLAG_IS_K_FULL = 1 << 2
FLAG_HAS_ZP = 1 << 3
FLAG_FORCE_SIMT = 1 << 8
FLAG_A_SMEM = 1 << 9
FLAG_FORCE_TC = 1 << 10
FLAG_FORCE_MMA = 1 << 11
FLAG_FORCE_SLICE = 1 << 13
FLAG_STATIC_WEIGHTS = 1 << 12

RTOL = 1e-2
ATOL = 1e-2


@dataclasses.dataclass
class Problem:
    m: int
    k: int
    n: int
    group_size: int
    weight_type: int
    a: np.ndarray            # fp16 [m, k]
    qweight: np.ndarray      # int32 [k/8, n] logical rows
    scales: np.ndarray       # fp16 [G, n]
    zeros: np.ndarray | None  # fp16 [G, n]
    g_idx: np.ndarray | None  # int32 [k]
    perm: np.ndarray | None   # int32 [k]

    @property
    def flags(self) -> int:
        f = FLAG_IS_K_FULL
        if self.zeros is not None:
            f |= FLAG_HAS_ZP
        if self.perm is not None:
            f |= FLAG_ACT_ORDER
        return f


def make_problem(seed: int, m: int, k: int, n: int, group_size: int = 128, weight_type: int = U4B8,
                 act_order: bool = False, sigma: float = 1.0) -> Problem:
    groups = synth.group_count(k, group_size)
    a = synth.activations(seed, m, k, sigma=sigma)
    qw = synth.qweight(seed, k, n)
    s = synth.scales(seed, groups, n)
    z = synth.zeros(seed, groups, n) if weight_type == U4 else None
    perm = g_idx = None
    if act_order:
        perm = synth.permutation(seed, k)
        g_idx = synth.act_order_gidx(perm, group_size if group_size != -1 else k)
    return Problem(m, k, n, group_size, weight_type, a, qw, s, z, g_idx, perm)


def oracle_ref(orc, pb: Problem, rows=None) -> np.ndarray:
    a = pb.a if rows is None else pb.a[rows]
    return orc.gemm(np.ascontiguousarray(a), pb.qweight, pb.scales, pb.zeros, pb.g_idx,
                    pb.group_size, pb.weight_type)


def within_tol(got: np.ndarray, ref: np.ndarray, rtol=RTOL, atol=ATOL):
    """Elementwise |got - ref| <= atol + rtol*|ref|, finite.  Returns (ok, message)."""
    got = np.asarray(got, dtype=np.float64)
    if got.shape != ref.shape:
        return False, f"shape {got.shape} vs {ref.shape}"
    if not np.all(np.isfinite(got)):
        return False, "non-finite output"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        return False, (f"{int(bad.sum())} of {bad.size} outside tolerance; first {idx}: "
                       f"{got[idx]} vs {ref[idx]} (max err {err.max():.3e})")
    return True, f"max err {err.max():.3e}"


# --- GPU side (imported lazily so the CPU suite never needs CUDA) ---------------------------

def torch_dev(x: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def repack_device(w4, qweight: np.ndarray, perm, k: int, n: int):
    import torch
    qw = torch_dev(qweight)
    out = torch.empty(k * n // 8, dtype=torch.int32, device="cuda")
    p = torch_dev(perm) if perm is not None else None
    w4.w4_repack(qw, p, out, k, n)
    return out


class DeviceProblem:
    """A problem's inputs on the device, with its packed weights and a zeroed workspace."""

    def __init__(self, w4, pb: Problem, flags_extra: int = 0):
        import torch
        self.w4 = w4
        self.pb = pb
        self.flags = pb.flags | flags_extra
        self.a = torch_dev(pb.a)
        self.b = repack_device(w4, pb.qweight, pb.perm, pb.k, pb.n)
        self.scales = torch_dev(pb.scales)
        self.zeros = torch_dev(pb.zeros) if pb.zeros is not None else None
        self.g_idx = torch_dev(pb.g_idx) if pb.g_idx is not None else None
        self.perm = torch_dev(pb.perm) if pb.perm is not None else None
        ws_bytes = w4.w4a16_workspace_size(pb.m, pb.n, pb.k, pb.group_size, self.flags)
        assert ws_bytes > 0
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        self.c = torch.empty((pb.m, pb.n), dtype=torch.float16, device="cuda")

    def run(self):
        pb = self.pb
        self.w4.w4a16_gemm(self.a, self.b, self.c, self.scales, self.zeros, self.g_idx, self.perm,
                           self.ws, pb.m, pb.n, pb.k, pb.group_size, pb.weight_type, self.flags)
        return self.c

    def result(self) -> np.ndarray:
        import torch
        torch.cuda.synchronize()
        return self.c.float().cpu().numpy().astype(np.float64)

    def status(self) -> int:
        return self.w4.w4a16_status(self.ws)

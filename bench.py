"""Benchmark of the W4A16 GEMM on GB300: one JSON line per run (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass over every GEMM of the workload.  The default workload, "all", is the whole
metric, M = 1..4096: the decode sweep (M in {1,4,8,16,32,64} x 4096x4096 and 4096x12288, u4b8),
prefill (M in {256,1024,4096} x 4096x11008 and 11008x4096, u4 + zeros), act-order (M in
{1,16,2048}, 8192x28672) and the grouped MoE pair (8 experts, 512 tokens top-2); the single
configurations remain selectable for profiling.  Inputs are seeded synthetic data already
resident in HBM.  Each GEMM of a step reads its own copy of the weights from a ring whose total
size is at least three times the L2 size: no step finds its weights in L2.  Steps are captured
once in a CUDA graph and timed with CUDA events on the launching stream, W untimed warm-up
steps first.

`value` is the step's fraction of roofline: the sum over its GEMMs of each GEMM's roofline
time max(bytes / HBM bandwidth, flops / dense fp16 tensor peak), over the measured step time.
`detail` gives every GEMM's own time, rates, bound and fraction (timed live, a graph of calls
per GEMM); `roofline` is the dominant kernel's (the one with the most time), from those times.

`--impl reference` times the CPU oracle instead (the only other place this script runs it):
each step is a bounded sample of the same workload, extrapolated per GEMM.

For N > 1 (torchrun) every rank runs the full workload on its own GPU (weak scaling, no
collective on the data path); value = all ranks' roofline time / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "W4A16 GEMM TFLOP/s and weight HBM GB/s vs M=1..4096 (fraction of roofline)"
U4, U4B8, FE4M3 = 4, 5, 8
FLAG_ACT_ORDER, FLAG_IS_K_FULL, FLAG_HAS_ZP = 1 << 1, 1 << 2, 1 << 3
# Inference weights are written once, long before the GEMMs that read them.
FLAG_STATIC_WEIGHTS = 1 << 12
W4A16_FLAG_BF16 = 1 << 16
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------------------------
# Workloads (the configurations of the W4A16 GEMM; shapes, distributions and seeds)
# ---------------------------------------------------------------------------------------------

CONFIGS = ("decode", "prefill", "actorder", "moe")


def workload_specs(name: str):
    """List of GEMMs of one step: dicts with m, k, n, gs, wt, act_order, sigma, seed (grouped
    GEMMs: n_exp, n_tok, top_k, pair_rows instead of m), each tagged with its configuration."""
    if name == "all":
        return [s for c in CONFIGS for s in workload_specs(c)]
    if name == "decode":
        specs = [dict(m=m, k=4096, n=n, gs=128, wt=U4B8, act_order=False, sigma=1.0, seed=1000 + m)
                 for n in (4096, 12288) for m in (1, 4, 8, 16, 32, 64)]
    elif name == "prefill":
        specs = [dict(m=m, k=k, n=n, gs=128, wt=U4, act_order=False, sigma=0.5, seed=2000 + m)
                 for (k, n) in ((4096, 11008), (11008, 4096)) for m in (256, 1024, 4096)]
    elif name == "actorder":
        specs = [dict(m=m, k=8192, n=28672, gs=128, wt=U4B8, act_order=True, sigma=1.0, seed=3000 + m)
                 for m in (1, 16, 2048)]
    elif name == "fp8":
        # FP8 E4M3 weights (W8A16), group 128, on the prefill FFN shape across M.
        specs = [dict(m=m, k=4096, n=11008, gs=128, wt=FE4M3, act_order=False, sigma=1.0, seed=6000 + m)
                 for m in (1, 16, 256, 1024, 4096)]
    elif name == "bf16":
        # BF16 activations, scales, zeros and output on the prefill FFN shape across M.
        specs = [dict(m=m, k=4096, n=11008, gs=128, wt=U4, act_order=False, sigma=0.5, seed=7000 + m,
                      bf16=True) for m in (1, 16, 256, 1024, 4096)]
    elif name == "tiny":
        specs = [dict(m=16, k=256, n=256, gs=128, wt=U4B8, act_order=False, sigma=1.0, seed=0)]
    elif name == "moe_swiglu":
        # The MoE FFN as two chained grouped calls: gate_up (2I = 28672 interleaved gate/up
        # columns) with the SwiGLU epilogue writing H [1024 pairs][14336], then down reading H.
        specs = [dict(grouped=True, n_exp=8, n_tok=512, top_k=2, k=4096, n=28672, gs=128, wt=U4B8,
                      seed=5000, pair_rows=False, glu=1),
                 dict(grouped=True, n_exp=8, n_tok=512, top_k=2, k=14336, n=4096, gs=128, wt=U4B8,
                      seed=5001, pair_rows=True, a_from=0)]
    elif name == "moe_blocks":
        # The MoE configuration through the vLLM block-routed interface (blocks of 64 rows),
        # the down projection scaling each pair row by its top-k weight.
        specs = [dict(grouped=True, n_exp=8, n_tok=512, top_k=2, k=4096, n=28672, gs=128, wt=U4B8,
                      seed=5000, pair_rows=False, blocks=64),
                 dict(grouped=True, n_exp=8, n_tok=512, top_k=2, k=14336, n=4096, gs=128, wt=U4B8,
                      seed=5001, pair_rows=True, blocks=64, mul_topk=True)]
    elif name == "moe":
        specs = [dict(grouped=True, n_exp=8, n_tok=512, top_k=2, k=4096, n=28672, gs=128, wt=U4B8,
                      seed=5000, pair_rows=False),
                 dict(grouped=True, n_exp=8, n_tok=512, top_k=2, k=14336, n=4096, gs=128, wt=U4B8,
                      seed=5001, pair_rows=True)]
    else:
        raise SystemExit(f"unknown workload {name}")
    for s in specs:
        s["config"] = name
    return specs


WORKLOAD_TEXT = {
    "decode": "decode sweep M in {1,4,8,16,32,64} x (K=4096,N=4096),(K=4096,N=12288), group 128, u4b8",
    "prefill": "prefill M in {256,1024,4096} x (K=4096,N=11008),(K=11008,N=4096), group 128, u4 + fp16 zeros",
    "actorder": "act-order M in {1,16,2048}, K=8192, N=28672, group 128, u4b8, shuffled g_idx",
    "tiny": "tiny M=16, K=256, N=256, group 128, u4b8",
    "bf16": ("BF16 activations/scales/zeros/output M in {1,16,256,1024,4096}, K=4096, N=11008, "
             "group 128, u4 + bf16 zeros"),
    "fp8": "FP8 E4M3 weights (W8A16) M in {1,16,256,1024,4096}, K=4096, N=11008, group 128, scales ~U[1e-4,2e-4]",
    "moe": "grouped MoE 8 experts, 512 tokens top-2, gate_up K=4096 N=28672 + down K=14336 N=4096, u4b8",
    "moe_blocks": ("grouped MoE 8 experts, 512 tokens top-2 through the vLLM block routing (blocks of "
                   "64 rows, sentinel padding): gate_up K=4096 N=28672 + down K=14336 N=4096 x top-k "
                   "weights, u4b8"),
    "moe_swiglu": ("grouped MoE FFN 8 experts, 512 tokens top-2: gate_up K=4096 2I=28672 with the "
                   "fused SwiGLU epilogue -> H [1024, 14336] -> down K=14336 N=4096 reading H, u4b8"),
}
WORKLOAD_TEXT["all"] = ("M=1..4096, every configuration in one step: " +
                        "; ".join(WORKLOAD_TEXT[c] for c in CONFIGS))


def weight_bytes(s) -> int:
    g = synth.group_count(s["k"], s["gs"])
    codes = s["k"] * s["n"] if s["wt"] == FE4M3 else s["k"] * s["n"] // 2
    return codes + g * s["n"] * 2 * (2 if s["wt"] == U4 else 1)


def gemm_bytes(s) -> int:
    """Algorithmic HBM bytes of one call: packed codes + scales (+ zeros) + A + C (+ g_idx, perm)."""
    b = weight_bytes(s) + s["m"] * s["k"] * 2 + s["m"] * s["n"] * 2
    if s.get("act_order"):
        b += 8 * s["k"]
    return b


def gemm_flops(s) -> int:
    return 2 * s["m"] * s["n"] * s["k"]


def grouped_accounting(s):
    """Bytes/flops of a grouped call: all experts' weights, gathered A, pair-major Y."""
    g = synth.group_count(s["k"], s["gs"])
    wb = s["n_exp"] * (s["k"] * s["n"] // 2 + g * s["n"] * 2)
    n_pairs = s["n_tok"] * s["top_k"]
    rows = n_pairs if s["pair_rows"] else s["n_tok"]
    n_out = s["n"] // 2 if s.get("glu") else s["n"]
    return wb, wb + rows * s["k"] * 2 + n_pairs * n_out * 2, 2 * n_pairs * s["n"] * s["k"]


def accounting(s):
    """(weight bytes, algorithmic bytes, flops) of one GEMM of a workload."""
    if s.get("grouped"):
        return grouped_accounting(s)
    return weight_bytes(s), gemm_bytes(s), gemm_flops(s)


def roofline_us(s, peaks):
    """The GEMM's roofline time in microseconds, max(bytes / HBM, flops / tensor peak), and
    which of the two bounds it ("hbm" or "tensor")."""
    _, b, f = accounting(s)
    t_hbm = b / peaks["hbm_gbs"] / 1e3
    t_tc = f / peaks["bf16_tflops"] / 1e6
    return (t_hbm, "hbm") if t_hbm >= t_tc else (t_tc, "tensor")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments, trailing blanks and empty lines."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments ignored): a recorded traffic figure stays
    valid across comment edits and lapses with any change to the code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_int4_03_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the hot-path kernels from the committed ncu summary
    (profiles/traffic.txt), or None if it is missing or was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 3 and not line.startswith("#") and parts[0] == workload:
                return int(parts[2]) if parts[1] == kernel_source_hash() else None
    return None


# ---------------------------------------------------------------------------------------------
# Multi-rank plumbing (also exercised by the gloo tests on CPU)
# ---------------------------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def aggregate_over_ranks(local_ms: float, local_units: float, group=None):
    """Max time and summed work over ranks (identity when torch.distributed is not up)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_ms, local_units
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------------------------------------
# Clock sampling
# ---------------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        window = [s for s in self.samples if t0 <= s[0] <= t1] or self.samples
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(p[1]) for _, p in window if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in window if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in window for i in range(4) if p[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(window)}


# ---------------------------------------------------------------------------------------------
# Our implementation
# ---------------------------------------------------------------------------------------------

class DenseGemm:
    """One dense GEMM of the workload with a ring of weight copies on the device."""

    def __init__(self, w4, s, copies: int, dev):
        import torch
        self.s = s
        k, n, m, gs = s["k"], s["n"], s["m"], s["gs"]
        groups = synth.group_count(k, gs)
        a = synth.activations(s["seed"], m, k, sigma=s["sigma"])
        fp8 = s["wt"] == FE4M3
        bf16 = bool(s.get("bf16"))
        qw = torch.from_numpy(synth.fp8_weights(s["seed"], k, n) if fp8 else
                              synth.qweight(s["seed"], k, n)).to(dev)
        perm = g_idx = None
        if s["act_order"]:
            p = synth.permutation(s["seed"], k)
            perm = torch.from_numpy(p).to(dev)
            g_idx = torch.from_numpy(synth.act_order_gidx(p, gs)).to(dev)
        if fp8:
            packed = torch.empty(k * n // 4, dtype=torch.int32, device=dev)
            w4.w8_repack(qw, packed, k, n)
        else:
            packed = torch.empty(k * n // 8, dtype=torch.int32, device=dev)
            w4.w4_repack(qw, perm, packed, k, n)
        del qw
        sc = synth.scales(s["seed"], groups, n, *((1e-4, 2e-4) if fp8 else ()))
        zr = synth.zeros(s["seed"], groups, n) if s["wt"] == U4 else None
        if bf16:   # the same values rounded to bfloat16, passed as raw 16-bit words
            a, sc = _bf16_words(a), _bf16_words(sc)
            zr = None if zr is None else _bf16_words(zr)
        scales = torch.from_numpy(sc).to(dev)
        zeros = torch.from_numpy(zr).to(dev) if zr is not None else None
        self.b = [packed] + [packed.clone() for _ in range(copies - 1)]
        self.scales = [scales] + [scales.clone() for _ in range(copies - 1)]
        self.zeros = None if zeros is None else [zeros] + [zeros.clone() for _ in range(copies - 1)]
        self.perm, self.g_idx = perm, g_idx
        self.flags = FLAG_IS_K_FULL | FLAG_STATIC_WEIGHTS | (FLAG_HAS_ZP if zeros is not None else 0) | (
            FLAG_ACT_ORDER if perm is not None else 0) | (W4A16_FLAG_BF16 if bf16 else 0)
        self.a_host = torch.from_numpy(a).pin_memory()
        self.a = self.a_host.to(dev)
        self.c = torch.empty((m, n), dtype=torch.int16 if bf16 else torch.float16, device=dev)
        self.ws = torch.zeros(w4.w4a16_workspace_size(m, n, k, gs, self.flags), dtype=torch.uint8,
                              device=dev)
        self.w4 = w4
        self.launches = 2 if perm is not None else 1

    def run(self, copy: int):
        s = self.s
        r = copy % len(self.b)
        self.w4.w4a16_gemm(self.a, self.b[r], self.c, self.scales[r],
                           None if self.zeros is None else self.zeros[r], self.g_idx, self.perm,
                           self.ws, s["m"], s["n"], s["k"], s["gs"], s["wt"], self.flags)

class GroupedGemm:
    """One grouped (MoE) GEMM over an expert-major CSR schedule."""

    def __init__(self, w4, s, copies: int, dev):
        import torch
        self.s = s
        n_exp, n_tok, top_k, k, n, gs = s["n_exp"], s["n_tok"], s["top_k"], s["k"], s["n"], s["gs"]
        groups = synth.group_count(k, gs)
        n_pairs = n_tok * top_k
        sel = synth.routes(5000, n_tok, n_exp, top_k)
        ex_ids, ex_off, ex_pairs, pair_tok = w4.w4a16_csr_from_token_routes(n_exp, n_tok, top_k, sel)
        rows = n_tok
        if s["pair_rows"]:   # down projection: pair-major activations, pair p reads row p
            rows = n_pairs
            pair_tok = np.arange(n_pairs, dtype=np.int32)
        self.blocks = s.get("blocks", 0)   # the vLLM block routing instead of the CSR schedule
        if self.blocks:
            # Down projection over pair rows: every pair is its own "token" with top_k 1.
            m_rows, tk = (n_tok, top_k) if not s["pair_rows"] else (n_pairs, 1)
            sid, eid, padded = w4.w4a16_moe_align_block_size(sel, m_rows, tk, n_exp, self.blocks)
            self.route = [torch.from_numpy(x).to(dev) for x in (sid, eid, np.array([padded], np.int32))]
            self.route_sizes = (padded, m_rows, tk)
            self.topk_w = (torch.from_numpy(synth.scales(s["seed"], 1, n_pairs, lo=0.05, hi=0.95)
                                            .astype(np.float32).ravel()).to(dev)
                           if s.get("mul_topk") else None)
        a = synth.activations(s["seed"], rows, k)
        glu = s.get("glu", 0)   # gated FFN: planar gate|up weights, interleaved on the device
        packed = torch.empty(n_exp * k * n // 8, dtype=torch.int32, device=dev)
        per = k * n // 8
        for e in range(n_exp):
            qw = torch.from_numpy(synth.qweight(s["seed"] * 100 + e, k, n)).to(dev)
            if glu:
                qw_i = torch.empty_like(qw)
                w4.w4_gate_up_interleave(qw, qw_i, k // 8, n)
                qw = qw_i
            w4.w4_repack(qw, None, packed[e * per:(e + 1) * per], k, n)
            del qw
        scales = torch.from_numpy(synth.scales(s["seed"], n_exp * groups, n)).to(dev)
        if glu:
            planar = scales
            scales = torch.empty_like(planar)
            w4.w4_gate_up_interleave(planar, scales, n_exp * groups, n)
            del planar
        self.b = [packed] + [packed.clone() for _ in range(copies - 1)]
        self.scales = [scales] + [scales.clone() for _ in range(copies - 1)]
        self.csr = [torch.from_numpy(x).to(dev) for x in (ex_ids, ex_off, ex_pairs, pair_tok)]
        self.n_active, self.n_pairs, self.rows = len(ex_ids), n_pairs, rows
        self.flags = FLAG_IS_K_FULL | (0 if not glu else w4.W4A16_FLAG_SWIGLU if glu == 1
                                       else w4.W4A16_FLAG_GEGLU)
        self.a_host = torch.from_numpy(a).pin_memory()
        self.a = self.a_host.to(dev)
        self.c = torch.empty((n_pairs, n // 2 if glu else n), dtype=torch.float16, device=dev)
        if self.blocks:
            ws_bytes = w4.w4a16_moe_blocks_workspace_size(self.route_sizes[0], self.blocks, n_exp, n,
                                                          k, gs, self.flags)
            self.launches = 3
        else:
            ws_bytes = w4.w4a16_grouped_workspace_size(n_pairs, self.n_active, n, k, gs, self.flags)
            self.launches = 2
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        self.w4 = w4
        s["m"] = n_pairs   # rows of output for the flop/byte accounting
        s["act_order"] = False
        s["sigma"] = 1.0

    def run(self, copy: int):
        s = self.s
        r = copy % len(self.b)
        if self.blocks:
            sid, eid, ntpp = self.route
            padded, m_rows, tk = self.route_sizes
            self.w4.w4a16_gemm_moe_blocks(self.a, self.b[r], self.c, self.scales[r], None, sid, eid,
                                          ntpp, self.topk_w, padded, self.blocks, tk,
                                          self.topk_w is not None, False, s["n_exp"], m_rows, s["n"],
                                          s["k"], s["gs"], s["wt"], self.flags, self.ws)
            return
        ids, off, pairs, tok = self.csr
        self.w4.w4a16_gemm_grouped(self.a, self.b[r], self.c, self.scales[r], None, ids, off, pairs, tok,
                                   self.n_active, s["n_exp"], self.n_pairs, self.rows, s["n"], s["k"],
                                   s["gs"], s["wt"], self.flags, self.ws)

class StepIO:
    """A step's activations in and results out for the end-to-end run: every GEMM's A and C
    in two device buffers (the step's parity picks one) and one pinned host buffer each, copied
    on two copy streams, one per direction: step s+1's inputs go up while step s computes, and
    step s's results come down behind it, while the next inputs go up.  (Each GEMM keeps
    tensors of its own: packing all of a step's A and C into one buffer changed nothing
    measurable; what cost 4 % on prefill was building this staging before the device-timed
    run, so bench builds it after.)"""

    def __init__(self, gemms, dev):
        import torch
        self.gemms = gemms
        # A GEMM whose A is an earlier GEMM's C (a chained FFN) reads that C in the same buffer
        # set and copies nothing in; a C that feeds a later GEMM is not copied out.
        self.src = [g.s.get("a_from") for g in gemms]
        fed = {i for i in self.src if i is not None}
        self.c_views = [[g.c for g in gemms], [torch.empty_like(g.c) for g in gemms]]
        self.a_views = [[g.a for g in gemms],
                        [g.a.clone() if i is None else None for g, i in zip(gemms, self.src)]]
        for b in range(2):
            for j, i in enumerate(self.src):
                if i is not None:
                    self.a_views[b][j] = self.c_views[b][i]
        self.copy_in = [i is None for i in self.src]
        self.copy_out = [j not in fed for j in range(len(gemms))]
        self.a_host = [g.a_host for g in gemms]
        self.c_host = [torch.empty(g.c.shape, dtype=g.c.dtype).pin_memory() if out else None
                       for g, out in zip(gemms, self.copy_out)]
        self.h2d_bytes = sum(g.a.numel() * 2 for g, cin in zip(gemms, self.copy_in) if cin)
        self.d2h_bytes = sum(g.c.numel() * 2 for g, out in zip(gemms, self.copy_out) if out)
        self.in_stream = torch.cuda.Stream(device=dev)
        self.out_stream = torch.cuda.Stream(device=dev)

    def h2d(self, b: int):
        for dst, src, cin in zip(self.a_views[b], self.a_host, self.copy_in):
            if cin:
                dst.copy_(src, non_blocking=True)

    def d2h(self, b: int):
        for dst, src, out in zip(self.c_host, self.c_views[b], self.copy_out):
            if out:
                dst.copy_(src, non_blocking=True)

    def bind(self, b: int):
        for g, a, c in zip(self.gemms, self.a_views[b], self.c_views[b]):
            g.a, g.c = a, c

    def enqueue_steps(self, stream, step0, nsteps, run_gemm):
        """Steps step0.. with their copies: h2d(s+1) overlaps step s, d2h(s) follows it.  The
        first step's GEMMs each wait only for their own inputs, and the last step's results
        each leave as soon as their GEMM is done (the pipeline's fill and drain are one GEMM's
        copy, not a whole step's).  run_gemm(st, j) runs GEMM j of step st."""
        import torch
        n = len(self.gemms)
        cin, cout = self.in_stream, self.out_stream
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]
        ev_in0 = [torch.cuda.Event() for _ in range(n)]
        ev_c = [torch.cuda.Event() for _ in range(n)]
        cin.wait_stream(stream)
        cout.wait_stream(stream)
        with torch.cuda.stream(cin):
            for j in range(n):
                if self.copy_in[j]:
                    self.a_views[0][j].copy_(self.a_host[j], non_blocking=True)
                    ev_in0[j].record(cin)
        for i in range(nsteps):
            b = i & 1
            last = i == nsteps - 1
            if i + 1 < nsteps:
                nb = (i + 1) & 1
                with torch.cuda.stream(cin):
                    if i >= 1:
                        cin.wait_event(ev_done[nb])   # step i-1 is done with buffer nb
                    self.h2d(nb)
                    ev_in[nb].record(cin)
            if i > 0:
                stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])         # step i-2's results have left buffer b
            self.bind(b)
            with torch.cuda.stream(stream):
                for j in range(n):
                    if i == 0 and self.copy_in[j]:
                        stream.wait_event(ev_in0[j])
                    run_gemm(step0 + i, j)
                    if last and self.copy_out[j]:
                        ev_c[j].record(stream)
                        with torch.cuda.stream(cout):
                            cout.wait_event(ev_c[j])
                            self.c_host[j].copy_(self.c_views[b][j], non_blocking=True)
            ev_done[b].record(stream)
            if not last:
                with torch.cuda.stream(cout):
                    cout.wait_event(ev_done[b])
                    self.d2h(b)
                    ev_out[b].record(cout)
        stream.wait_stream(cin)
        stream.wait_stream(cout)
        self.bind(0)


def select_shape(specs, shape):
    """The GEMMs of `specs` whose (m, k, n) equal the "M,K,N" string `shape` (all if None)."""
    if not shape:
        return specs
    m, k, n = (int(v) for v in shape.split(","))
    picked = [s for s in specs if (s.get("m"), s["k"], s["n"]) == (m, k, n)]
    if not picked:
        raise SystemExit(f"no GEMM {shape} in this workload")
    return picked


def time_graph(stream, dev, fn, reps):
    """Average microseconds of one fn(r) call, from a CUDA graph of `reps` calls (r = 0..reps-1)
    timed with CUDA events on `stream` after one warm replay."""
    import torch
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn(0)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(graph, stream=stream):
            for r in range(reps):
                fn(r)
        graph.replay()
    torch.cuda.synchronize(dev)
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    with torch.cuda.stream(stream):
        graph.replay()
    d1.record(stream)
    torch.cuda.synchronize(dev)
    del graph
    return d0.elapsed_time(d1) * 1e3 / reps


def kernel_of(w4, g) -> int:
    """The library's kernel for one GEMM of the workload (0 tcgen05, 1 split-K small-M,
    2 column-slice small-M); grouped calls always run the tcgen05 kernel."""
    s = g.s
    if s.get("grouped"):   # grouped calls: always tcgen05
        return 0
    if s["wt"] == FE4M3:   # FP8: the column-slice kernel up to 16 tokens, else tcgen05
        import torch
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        return 2 if s["m"] <= 16 and s["n"] // 16 >= sms else 0
    return w4.w4a16_kernel_for(s["m"], s["n"], s["k"], s["gs"], g.flags)


def kernel_roofline(rows, peaks, peak_src, launches):
    """Roofline of one kernel from the live per-GEMM timings of its calls: the bound its calls'
    roofline times are mostly set by, achieved = their algorithmic flops (bytes) / their time."""
    us = sum(r["us"] for r in rows)
    flops = sum(r["flops"] for r in rows)
    nbytes = sum(r["bytes"] for r in rows)
    t_tc = sum(r["roof_us"] for r in rows if r["bound"] == "tensor")
    t_hbm = sum(r["roof_us"] for r in rows if r["bound"] == "hbm")
    if t_tc >= t_hbm:
        achieved = flops / us / 1e6
        out = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
               "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
               "peak_source": f"{peak_src} bf16_tflops (burst; the fp16 dense rate equals bf16)",
               "flops_per_launch": round(flops / launches)}
    else:
        achieved = nbytes / us / 1e3
        out = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
               "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
               "peak_source": f"{peak_src} hbm_gbs", "bytes_per_launch": round(nbytes / launches)}
    out["launches_per_step"] = launches
    out["us_per_step"] = round(us, 2)
    return out


def run_ours(args, rank, world, local):
    import torch
    import weight_only_int4_03_gb300 as w4

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 1024 * 1024
    peaks, peak_src = load_peaks()
    specs = select_shape(workload_specs(args.workload), args.shape)
    gemms = []
    for s in specs:
        wb = accounting(s)[0]
        copies = max(1, min(64, math.ceil(3 * l2 / wb)))
        gemms.append(GroupedGemm(w4, s, copies, dev) if s.get("grouped") else DenseGemm(w4, s, copies, dev))
    for g in gemms:   # chained FFN: this GEMM's A is an earlier GEMM's output
        if g.s.get("a_from") is not None:
            src = gemms[g.s["a_from"]].c
            assert src.shape == g.a.shape, (src.shape, g.a.shape)
            g.a = src

    # Per-step accounting: algorithmic bytes and flops, and the roofline time of every GEMM.
    step_wbytes = step_bytes = step_flops = 0
    step_roof_us = 0.0
    for g in gemms:
        wb, b, f = accounting(g.s)
        step_wbytes += wb
        step_bytes += b
        step_flops += f
        step_roof_us += roofline_us(g.s, peaks)[0]
    launches_per_step = sum(g.launches for g in gemms)

    stream = torch.cuda.Stream(device=dev)
    io = None   # the end-to-end staging, built after the device-timed run

    def run_gemm(st, gi):
        gemms[gi].run(st * len(gemms) + gi)

    def run_step(st):
        for gi in range(len(gemms)):
            run_gemm(st, gi)

    def enqueue(step0, nsteps, e2e=False):
        if e2e:
            io.enqueue_steps(stream, step0, nsteps, run_gemm)
            return
        for st in range(step0, step0 + nsteps):
            run_step(st)

    # Eager warm-up of every code path (also initialises the library's per-device state).
    with torch.cuda.stream(stream):
        enqueue(0, 1)
    torch.cuda.synchronize(dev)
    for g in gemms:
        bits = w4.w4a16_status(g.ws, stream=stream)
        if bits:
            raise SystemExit(f"device status {bits} after warm-up")

    def capture(step0, nsteps, e2e=False):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                enqueue(step0, nsteps, e2e)
        return graph

    warm_graph = capture(0, args.warmup)
    timed_graph = capture(args.warmup, args.steps)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    import torch.distributed as dist
    distributed = dist.is_available() and dist.is_initialized()
    with torch.cuda.stream(stream):
        warm_graph.replay()
    torch.cuda.synchronize(dev)
    if distributed:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    with torch.cuda.stream(stream):
        timed_graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if distributed:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    # Keep the GPU busy briefly so the clock record has samples under the same load.
    t_tail = time.time()
    while time.time() - t_tail < 0.6:
        with torch.cuda.stream(stream):
            timed_graph.replay()
        torch.cuda.synchronize(dev)
    clocks.stop()
    clk = clocks.summary(t_wall0 - 0.35, time.time())
    del warm_graph, timed_graph

    # End to end: every step's A in from pinned host memory and C out, inside the timed
    # region.  The staging (a second set of device buffers, a copy stream) is made only now:
    # allocated before the device-timed run it slowed the prefill kernels by 4 %.
    io = StepIO(gemms, dev)
    e2e_graph = capture(args.warmup, args.steps, e2e=True)
    with torch.cuda.stream(stream):
        e2e_graph.replay()
    torch.cuda.synchronize(dev)
    if distributed:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        e2e_graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    del e2e_graph

    for g in gemms:
        bits = w4.w4a16_status(g.ws, stream=stream)
        if bits:
            raise SystemExit(f"device status {bits} after timing")

    # value: the step's roofline time over its measured time (summed over ranks' work).
    roof_units = step_roof_us * 1e-3 * args.steps          # ms of roofline time
    max_ms, all_roof = aggregate_over_ranks(ms, roof_units)
    max_e2e, all_roof_e2e = aggregate_over_ranks(e2e_ms, roof_units)

    # Per-GEMM detail, timed live (graphs of R calls of one GEMM over its weight ring): each
    # GEMM's time, rates and roofline fraction, and which kernel ran it.  The roofline of the
    # dominant kernel is computed from these times.
    detail = []
    if rank == 0 and not args.no_detail:
        for g in gemms:
            wb, b, f = accounting(g.s)
            reps = max(20, min(200, int(2e8 / max(1, wb))))
            us = time_graph(stream, dev, g.run, reps)
            roof, bound = roofline_us(g.s, peaks)
            kern = kernel_of(w4, g)
            row = {"config": g.s["config"], "m": g.s["m"], "k": g.s["k"], "n": g.s["n"],
                   "kernel": w4.KERNEL_NAMES[kern], "us": round(us, 3),
                   "tflops": round(f / us * 1e-6, 2), "weight_gbs": round(wb / us * 1e-3, 1),
                   "bytes_gbs": round(b / us * 1e-3, 1), "bound": bound,
                   "roof_us": round(roof, 3), "frac": round(roof / us, 4)}
            if g.s.get("grouped"):
                row["experts"] = g.s["n_exp"]
            detail.append(row)
            row["_flops"], row["_bytes"], row["_launches"], row["_kern"] = f, b, g.launches, kern

    if rank != 0:
        return None
    sec = max_ms * 1e-3
    by_kernel = {}
    for r in detail:
        by_kernel.setdefault(r["_kern"], []).append(
            {"us": r["us"], "flops": r["_flops"], "bytes": r["_bytes"], "roof_us": r["roof_us"],
             "bound": r["bound"], "launches": r["_launches"]})
    kernels = {}
    for kern, rows in by_kernel.items():
        launches = sum(x["launches"] for x in rows)
        kr = kernel_roofline(rows, peaks, peak_src, launches)
        key = f"{args.workload}:{w4.KERNEL_NAMES[kern].split()[0]}"
        kr["traffic"] = recorded_traffic(key) if not args.shape else None
        kernels[w4.KERNEL_NAMES[kern]] = kr
    dominant = max(kernels, key=lambda name: kernels[name]["us_per_step"]) if kernels else None
    roof = dict(kernels[dominant], kernel=dominant) if dominant else None
    for r in detail:
        for key in ("_flops", "_bytes", "_launches", "_kern"):
            r.pop(key)
    value = all_roof / max_ms
    e2e_value = all_roof_e2e / max_e2e
    unit = "fraction of roofline (sum over the step's GEMMs of max(bytes/HBM, flops/tensor peak) / step time)"
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": _dtype_text(specs),
        "data": "synthetic (seeded LCG; shapes and distributions of the W4A16 configurations)",
        "config": {"workload": WORKLOAD_TEXT[args.workload] + (f" (only {args.shape})" if args.shape else ""),
                   "gemms_per_step": len(gemms),
                   "l2_defeat": "weight-copy ring >= 3x L2 per shape", "graph": "CUDA graph of all steps",
                   "parallelism": f"replicas x{world}"},
        "tflops": round(step_flops * args.steps / sec / 1e12, 2),
        "weight_gbs": round(step_wbytes * args.steps / sec / 1e9, 1),
        "roofline_us_per_step": round(step_roof_us, 2),
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "tensor_tflops": peaks["bf16_tflops"],
                  "source": peak_src},
        "roofline": roof,
        "kernels": kernels,
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 4), "unit": unit, "h2d_bytes_per_step": io.h2d_bytes,
                "d2h_bytes_per_step": io.d2h_bytes, "ms_per_step": round(max_e2e / args.steps, 5),
                "mode": "C ABI calls; every GEMM's A in from pinned host memory and C out, on two copy streams (one per direction) overlapping the neighbouring steps' compute (double-buffered), captured in a CUDA graph"},
        "gpu_launches": launches_per_step * args.steps,
        "detail": detail,
    }
    return line


# ---------------------------------------------------------------------------------------------
# The oracle (CPU) as a reported baseline and as the reference arm
# ---------------------------------------------------------------------------------------------

def _dtype_text(specs) -> str:
    acts = "bf16" if any(s.get("bf16") for s in specs) else "f16"
    codes = "/".join(sorted({"e4m3" if s["wt"] == FE4M3 else "u4" for s in specs}))
    return f"{acts} x {codes} -> f32 acc"


def _bf16_words(x):
    """int16 words of the bfloat16 roundings of an array's values."""
    return synth.bf16_bits(np.asarray(x, dtype=np.float64)).view(np.int16)


def _bf16_values(words):
    return (np.asarray(words).view(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _oracle_inputs(s, rows: int):
    """Oracle inputs of one GEMM of the workload with `rows` activation rows (for a grouped
    GEMM: one expert's weights, rows standing for (token, expert) pairs)."""
    k, n = s["k"], s["n"]
    g = synth.group_count(k, s["gs"])
    if s.get("grouped"):
        qw = synth.qweight(s["seed"] * 100, k, n)
        a = synth.activations(s["seed"], rows, k)
        return a, qw, synth.scales(s["seed"], g, n), None, None
    if s["wt"] == FE4M3:
        return (synth.activations(s["seed"], rows, k, sigma=s["sigma"]), synth.fp8_weights(s["seed"], k, n),
                synth.scales(s["seed"], g, n, 1e-4, 2e-4), None, None)
    qw = synth.qweight(s["seed"], k, n)
    z = synth.zeros(s["seed"], g, n) if s["wt"] == U4 else None
    g_idx = synth.act_order_gidx(synth.permutation(s["seed"], k), s["gs"]) if s.get("act_order") else None
    a, sc = synth.activations(s["seed"], rows, k, sigma=s["sigma"]), synth.scales(s["seed"], g, n)
    if s.get("bf16"):
        a, sc = _bf16_words(a), _bf16_words(sc)
        z = None if z is None else _bf16_words(z)
    return a, qw, sc, z, g_idx


def step_totals(specs, peaks):
    """(roofline microseconds, flops, weight bytes) of one step of these GEMMs."""
    roof = flops = wbytes = 0.0
    for s in specs:
        wb, _, f = accounting(s)
        roof += roofline_us(s, peaks)[0]
        flops += f
        wbytes += wb
    return roof, flops, wbytes


def oracle_sample(workload: str, budget_s: float, threads: int | None = None):
    """Times the oracle on a bounded sample of one step of the workload and estimates the time
    of the whole step.  The oracle derives W once per call (a fixed cost) and then spends a
    fixed time per output row, so every GEMM is timed at 1 row and at r rows (r sized from the
    budget) and the two-point fit extrapolates to all of its rows (a grouped GEMM pays the W
    derivation once per expert).
    Returns (step_seconds_estimate, threads, sample_text)."""
    import oracle
    orc = oracle.Oracle()
    threads = threads or oracle.default_threads()
    specs = workload_specs(workload)

    def seconds(s, r):
        a, qw, sc, z, g_idx = _oracle_inputs(s, r)
        t0 = time.perf_counter()
        if s["wt"] == FE4M3:
            orc.gemm_fp8(a, qw, sc, s["gs"], threads=threads)
        elif s.get("bf16"):
            orc.gemm_bf16(a.view(np.uint16), qw, sc.view(np.uint16),
                          None if z is None else z.view(np.uint16), g_idx, s["gs"], s["wt"], threads=threads)
        else:
            orc.gemm(a, qw, sc, z, g_idx, s["gs"], s["wt"], threads=threads)
        return time.perf_counter() - t0

    per_gemm = budget_s / max(1, len(specs))
    est = 0.0
    sample_rows = 0
    for s in specs:
        rows_total = s["n_tok"] * s["top_k"] if s.get("grouped") else s["m"]
        fixed_count = s["n_exp"] if s.get("grouped") else 1
        t1 = seconds(s, 1)
        sample_rows += 1
        # A row costs roughly a twentieth of deriving W (one multiply-add per weight against
        # the weight's full derivation); the second point then measures it.
        r = int(min(rows_total, 4096, max(2, (per_gemm - t1) / max(t1 / 20, 1e-9))))
        if rows_total > 1 and r >= 2:
            tr = seconds(s, r)
            sample_rows += r
            per_row = max(0.0, (tr - t1) / (r - 1))
            fixed = max(0.0, t1 - per_row)
        else:
            per_row, fixed = t1, 0.0
        est += fixed_count * fixed + rows_total * per_row
    text = (f"{sample_rows} output rows over the {len(specs)} GEMMs of one step (each GEMM at 1 "
            f"row and at up to 4096 rows), fp64 on {threads} threads; the step time is the "
            f"two-point fit (W derivation + rows x per-row time) summed over the GEMMs")
    return est, threads, text


def _dequant_fp8_fp32(qw, scales, gs):
    """[K][N] fp32 weights e4m3(code) * s from [K/4][N] words of four K-consecutive codes (row
    4r+i at byte i), decoded by torch's float8_e4m3fn, for the BLAS baseline."""
    import torch
    k4, n = qw.shape
    codes = qw.view(np.uint8).reshape(k4, n, 4).transpose(0, 2, 1).reshape(k4 * 4, n)
    w = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).float().numpy()
    k = k4 * 4
    g = np.arange(k) // (gs if gs > 0 else k)
    return w * scales.astype(np.float32)[g]


def _dequant_fp32(qw, scales, zeros, gs, wt):
    """[K][N] fp32 weights (q - z) * s from GPTQ words (row 8r+i at bits 4i..4i+3), for the
    BLAS baseline; z = 8 for u4b8."""
    k8, n = qw.shape
    q = np.empty((k8 * 8, n), dtype=np.float32)
    w = qw.view(np.uint32)
    for i in range(8):
        q[i::8] = ((w >> np.uint32(4 * i)) & np.uint32(0xF)).astype(np.float32)
    k = k8 * 8
    g = np.arange(k) // (gs if gs > 0 else k)
    s = scales.astype(np.float32)[g]
    z = zeros.astype(np.float32)[g] if wt == U4 else np.float32(8.0)
    q -= z
    q *= s
    return q


def blas_sample(workload: str, repeats: int = 3):
    """A CPU baseline that is not the oracle: each GEMM's weights dequantised once to fp32
    (outside the timing), then numpy's fp32 GEMM (BLAS, the host's threads) on the GEMM's full
    M, best of `repeats`.  For a grouped GEMM one expert's weights stand for every expert and
    the time is scaled by the experts.  Returns (step_seconds, text)."""
    est = 0.0
    specs = workload_specs(workload)
    for s in specs:
        rows = s["n_tok"] * s["top_k"] if s.get("grouped") else s["m"]
        per = rows // s["n_exp"] if s.get("grouped") else rows
        a, qw, sc, z, _ = _oracle_inputs(s, per)
        if s.get("bf16"):
            a, sc = _bf16_values(a), _bf16_values(sc)
            z = None if z is None else _bf16_values(z)
        w = _dequant_fp8_fp32(qw, sc, s["gs"]) if s["wt"] == FE4M3 else _dequant_fp32(qw, sc, z, s["gs"], s["wt"])
        a32 = a.astype(np.float32)
        best = float("inf")
        for _ in range(repeats):
            t0 = time.perf_counter()
            (a32 @ w).astype(np.float16)
            best = min(best, time.perf_counter() - t0)
        est += best * (s["n_exp"] if s.get("grouped") else 1)
        del w, a32
    text = (f"all {len(specs)} GEMMs of one step at full M, weights dequantised once to fp32 "
            f"outside the timing, numpy fp32 matmul (BLAS), best of {repeats}")
    return est, text


def cpu_line(workload: str, seconds: float, peaks):
    """A CPU step time in the line's units: the step's roofline time on the GPU over the CPU's
    step time (the same fraction the GPU line reports), plus TFLOP/s and weight GB/s."""
    roof, flops, wbytes = step_totals(workload_specs(workload), peaks)
    return {"value": round(roof * 1e-6 / seconds, 8),
            "unit": "fraction of the GPU roofline (the step's roofline time / the CPU step time)",
            "tflops": round(flops / seconds / 1e12, 6), "weight_gbs": round(wbytes / seconds / 1e9, 6),
            "step_s": round(seconds, 3)}


def cpu_baseline(workload: str, budget_s: float = 15.0):
    """The oracle on the host's threads (the reported baseline), plus, labelled separately, the
    oracle on one thread and a BLAS fp32 GEMM on weights dequantised once.  The two extras are
    best effort: a failure is recorded in the line, it does not end the run."""
    peaks = load_peaks()[0]
    est, threads, text = oracle_sample(workload, budget_s)
    line = dict(cpu_line(workload, est, peaks), cores=threads, kind="oracle", sample=text)
    try:
        est1, _, text1 = oracle_sample(workload, budget_s / 3, threads=1)
        line["single_core"] = dict(cpu_line(workload, est1, peaks), cores=1, sample=text1)
    except Exception as e:  # noqa: BLE001 -- a baseline must not end the benchmark
        line["single_core"] = {"error": f"{type(e).__name__}: {e}"}
    try:
        est2, text2 = blas_sample(workload)
        line["fp32_blas"] = dict(cpu_line(workload, est2, peaks), cores=os.cpu_count(),
                                 kind="numpy fp32 GEMM on dequantised weights", sample=text2)
    except Exception as e:  # noqa: BLE001
        line["fp32_blas"] = {"error": f"{type(e).__name__}: {e}"}
    return line


def run_reference(args, rank):
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    per_step_budget = max(0.5, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(args.workload, per_step_budget)
    total_est = 0.0
    wall0 = time.time()
    threads = 1
    text = ""
    for _ in range(args.steps):
        est, threads, text = oracle_sample(args.workload, per_step_budget)
        total_est += est
    wall = time.time() - wall0
    cl = cpu_line(args.workload, total_est / args.steps, peaks)
    return {
        "impl": "reference", "metric": METRIC, "value": cl["value"], "unit": cl["unit"], "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_est / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded LCG)", "config": {"workload": WORKLOAD_TEXT[args.workload],
                                                     "parallelism": "CPU threads"},
        "tflops": cl["tflops"], "weight_gbs": cl["weight_gbs"],
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "tensor_tflops": peaks["bf16_tflops"], "source": peak_src},
        "cpu_baseline": {"value": cl["value"], "unit": cl["unit"], "cores": threads, "kind": "oracle",
                         "sample": text},
        "e2e": {"value": cl["value"], "unit": cl["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 2),
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOAD_TEXT), default="all")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-detail", action="store_true",
                    help="skip the per-GEMM timings (and with them the kernel rooflines): for profiling runs")
    ap.add_argument("--shape", default=None,
                    help="M,K,N: run only this GEMM of the workload (for profiling one kernel)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_env()

    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    import torch
    import torch.distributed as dist
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        line = run_ours(args, rank, world, local)
    finally:
        if world > 1 and dist.is_initialized():
            dist.destroy_process_group()
    if line is not None:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload)
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())

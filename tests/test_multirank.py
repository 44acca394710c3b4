"""The N>1 path of bench.py on CPU: two gloo ranks (replicas, no data-path collective).

Each rank runs the same workload on its own GPU in a real run; the only cross-rank steps are
the barrier around the timed region and the reduction of the result (max time, summed work).
These tests exercise that host logic with world_size 2 over gloo, and the workload accounting
that feeds it.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        dist.barrier()
        # Rank r "took" 10 + r ms for 100 * (r + 1) units of work.
        ms, units = bench.aggregate_over_ranks(10.0 + rank, 100.0 * (rank + 1))
        out[rank] = (ms, units)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_summed_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: (11.0, 300.0), 1: (11.0, 300.0)}


def test_single_process_aggregate_is_identity():
    assert bench.aggregate_over_ranks(3.5, 42.0) == (3.5, 42.0)


def test_workload_accounting():
    """Bytes and flops of the decode sweep follow the algorithmic definitions."""
    specs = bench.workload_specs("decode")
    assert len(specs) == 12
    s = next(x for x in specs if (x["m"], x["k"], x["n"]) == (1, 4096, 4096))
    # codes K*N/2 + scales G*N*2 (G = 32) + A M*K*2 + C M*N*2
    assert bench.weight_bytes(s) == 4096 * 4096 // 2 + 32 * 4096 * 2
    assert bench.gemm_bytes(s) == bench.weight_bytes(s) + 4096 * 2 + 4096 * 2
    assert bench.gemm_flops(s) == 2 * 4096 * 4096
    p = next(x for x in bench.workload_specs("prefill") if x["m"] == 256 and x["k"] == 11008)
    # u4 adds the zero points: G = 86 rows of N fp16 values
    assert bench.weight_bytes(p) == 11008 * 4096 // 2 + 2 * 86 * 4096 * 2
    moe = bench.workload_specs("moe")[0]
    wb, b, f = bench.grouped_accounting(moe)
    assert wb == 8 * (4096 * 28672 // 2 + 32 * 28672 * 2)
    assert f == 2 * 1024 * 28672 * 4096


def test_shape_filter():
    specs = bench.workload_specs("decode")
    assert len(bench.select_shape(specs, None)) == 12
    picked = bench.select_shape(specs, "16,4096,12288")
    assert len(picked) == 1 and picked[0]["m"] == 16
    with pytest.raises(SystemExit):
        bench.select_shape(specs, "3,4096,4096")

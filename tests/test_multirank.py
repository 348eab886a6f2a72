"""The benchmark's multi-rank path (one process per GPU, replicas with no
collective on the data path) on CPU with the gloo backend, world size 2: the
step time is the max over ranks, the throughput counts every rank's work,
and only rank 0 reports."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier()
        # rank 1 is the slow one: 4 ms per step vs 2 ms
        ms = 2.0 * (rank + 1)
        value, ms_max = bench.whole_job_tflops(1e12, ms, ws)
        out[rank] = (value, ms_max, bench.max_over_ranks(float(rank)))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_with_gloo():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        value, ms_max, mx = out[r]
        assert ms_max == 4.0          # slowest rank
        assert mx == 1.0
        # 2 ranks x 1 TFLOP in 4 ms = 500 TFLOP/s
        assert abs(value - 500.0) < 1e-9


def test_reference_arm_only_rank0_reports(monkeypatch):
    import bench
    from workloads import WORKLOADS

    class Args:
        steps, warmup, cpu_budget = 1, 3, 1.0

    assert bench.run_reference(Args, WORKLOADS["single_head_fp32"], 2, 1) is None
    line = bench.run_reference(Args, WORKLOADS["single_head_fp32"], 1, 0)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"

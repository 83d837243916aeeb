"""The multi-GPU bench path is replicas only: one process per GPU, no data-path collective.
Its host-side logic -- the barrier, the step time as the max over ranks, the throughput as the
sum over ranks, the reference arm printing on rank 0 only -- runs here as two gloo ranks on
the CPU."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier()
        ms = [3.0, 5.0][rank]              # per-rank step times
        step_ms = bench.reduce_max(ms)
        value = bench.reduce_sum(1000.0 / ms)  # each replica's throughput, summed
        buf = io.StringIO()

        class Args:
            workload, steps, warmup = "tiny", 1, 1

        with contextlib.redirect_stdout(buf):
            bench.run_reference(Args, rank, world)
        results[rank] = (step_ms, value, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_two_replicas_on_gloo():
    pytest.importorskip("numpy")
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), results), nprocs=world,
                           start_method="spawn")
        results = dict(results)
    for rank in range(world):
        step_ms, value, out = results[rank]
        assert step_ms == 5.0                       # the slowest replica sets the step time
        assert value == pytest.approx(1000 / 3 + 1000 / 5)
    assert '"impl": "reference"' in results[0][2] and '"n_gpus": 2' in results[0][2]
    assert results[1][2] == ""                      # other ranks print nothing

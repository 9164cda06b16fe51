"""The multi-GPU path of bench.py on the CPU: independent replicas over a world-size-2 gloo group.

One sequence at batch 1 is a serial chain of steps, so several GPUs run independent replicas
with no data exchange; only the timing is combined: the time is the maximum over ranks and the
whole-job value counts every rank's tokens.  The reference arm runs on rank 0 alone.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms, value = bench.aggregate_replicas(100.0 * (rank + 1), 256, world, "cpu")
        args = type("A", (), {"workload": "tiny", "steps": 1, "warmup": 0})()
        ref = bench.run_reference(args, rank, world) if rank != 0 else "skipped"
        out[rank] = (ms, value, ref)
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, value, _ = res[rank]
        assert ms == 200.0                                  # the slower rank's time on every rank
        assert value == pytest.approx(2 * 256 / 0.2)        # both ranks' tokens over that time
    assert res[1][2] is None                                # the reference arm: rank 0 alone


def test_single_rank_needs_no_group():
    import bench
    ms, value = bench.aggregate_replicas(50.0, 100, 1, "cpu")
    assert ms == 50.0 and value == pytest.approx(2000.0)

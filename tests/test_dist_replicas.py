"""The N > 1 bench path on CPU: two gloo ranks (127.0.0.1), as torchrun launches
them.  Each rank processes its own replica; the job time is the slowest rank's
and the whole-job throughput counts every rank's units.  The reference arm runs
on rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.env_rank()
        assert (r, lr, w) == (rank, rank, world)
        dist.barrier()
        slowest = bench.max_over_ranks(times[rank], dist, device="cpu")
        out[rank] = (slowest, bench.replica_throughput(16384, w, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [0.40, 0.55]
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        slowest, value = res[rank]
        assert slowest == pytest.approx(0.55)
        # every rank's 16384 tokens over the slowest rank's time
        assert value == pytest.approx(2 * 16384 / 0.55e-3)


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(0.3, None) == 0.3
    assert bench.replica_throughput(100, 1, 2.0) == pytest.approx(5e4)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        config = "uniform_8x2048"
        steps = 1
        warmup = 0
    bench.run_reference(Args(), rank=1, world=2)   # returns at once, prints nothing
    assert capsys.readouterr().out == ""

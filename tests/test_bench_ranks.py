"""Host logic of the benchmark's multi-rank path, on CPU ranks (gloo).

One process per GPU runs its own replica (the path shards by request and by
head with no exchange); the job's throughput is every rank's bytes over the
slowest rank's time.  Here two gloo ranks stand in for two GPUs.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.reduce_max(times[rank], dist, "cpu")
        out[rank] = (m, bench.whole_job_gbs(1e6, m, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [10.0, 12.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        m, gbs = res[rank]
        assert m == pytest.approx(12.5)
        assert gbs == pytest.approx(2 * 1e6 / 12.5e-6 / 1e9)


def test_single_rank_is_the_identity():
    assert bench.reduce_max(3.5, None, "cpu") == 3.5
    assert bench.whole_job_gbs(101646336, 17.9, 1) == pytest.approx(101646336 / 17.9e-6 / 1e9)


def test_reference_arm_other_ranks_do_nothing(capsys):
    class Args:
        steps, gpus = 2, 2
    assert bench.run_reference(Args(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""


def test_reference_sample_size_bounds():
    assert bench.reference_sample_size(20000, 2.7e-3) == 64      # 54 s for whole steps
    assert bench.reference_sample_size(20000, 27e-3) == 7        # 64 * 60 / 540
    assert bench.reference_sample_size(10, 2.7e-3) == 64
    assert bench.reference_sample_size(10**9, 1.0) == 1

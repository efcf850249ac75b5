"""The benchmark's multi-rank plumbing on CPU: two gloo ranks, each with its
own replica timing, agree on the max over ranks (the path has no exchange
between GPUs, so replicas are the only multi-GPU mode)."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench._dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(world)
    t = bench.aggregate_max(10.0 + 5.0 * rank, world)
    results[rank] = t
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        assert dict(results) == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate_max(3.5, 1) == 3.5


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.main.__globals__["argparse"].Namespace(config="tiny_none", steps=1, warmup=3, gpus=2)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""

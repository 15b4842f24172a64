"""The benchmark's multi-rank bookkeeping on CPU ranks (gloo, world size 2):
time is the max over ranks, throughput sums the replicas' work, and a rank
that is not rank 0 prints nothing for the reference arm."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.0 + rank * 0.5)
        w, r, lr = bench.dist_env()
        out[rank] = (t, w, r, lr)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_env_gloo():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0][0] == 1.5 and out[1][0] == 1.5
    assert [out[r][1:] for r in range(world)] == [(2, 0, 0), (2, 1, 1)]


def test_single_rank_identity_and_throughput():
    assert bench.max_over_ranks(3.25) == 3.25
    flop = 2 * 37810 * 5376 * 14336
    one = bench.job_throughput(1, flop, 2e-3)
    assert bench.job_throughput(4, flop, 2e-3) == pytest.approx(4 * one)
    assert one == pytest.approx(flop / 2e-3 / 1e12)


def test_reference_arm_silent_on_other_ranks(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), {"gpus": 2, "steps": 1, "warmup": 3})()
    bench.run_reference(args)
    assert capsys.readouterr().out == ""

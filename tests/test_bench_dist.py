"""bench.py's multi-rank plumbing on CPU: two gloo ranks, as torchrun would
launch them, agree on the slowest rank's time (max over ranks)."""

import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    out[rank] = bench.max_over_ranks(1.5 + rank, ws)
    bench.barrier(ws)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("LOCAL_RANK", raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_runs_on_rank_zero_only(capsys):
    """Under torchrun the reference arm prints from rank 0; other ranks exit without work."""
    import argparse
    args = argparse.Namespace(steps=1, warmup=3)
    assert bench.run_reference(args, 2, 1) is None
    assert capsys.readouterr().out == ""

"""Host logic of bench.py's multi-rank ("replicas only") mode, on CPU with
two gloo ranks: the timed region is the maximum over ranks, the rate counts
the units of all ranks, and the reference arm runs on rank 0 alone."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "took" 1.5 + r seconds: every rank must see the slowest
        t = bench.max_over_ranks(1.5 + rank, "cpu")
        out[rank] = (t, bench.whole_job_rate(dist.get_world_size(), 30, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rate_with_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    for t, rate in res.values():
        assert t == 2.5
        assert rate == pytest.approx(2 * 30 / 2.5)


def test_single_process_max_is_identity_and_rate():
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.whole_job_rate(1, 10, 2.0) == 5.0
    assert bench.whole_job_rate(4, 10, 2.0) == 20.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""

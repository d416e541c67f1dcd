"""The multi-rank path of bench.py on the CPU: two gloo ranks, each with its own step time.

The bench launches one process per GPU; every rank processes its own megabatches (weak
scaling, no collective on the data path).  These tests check, without a GPU, the host logic
around that: the slowest rank's time is what every rank reports, the whole-job figure divides
it by the number of ranks, ranks draw disjoint seeds, and the reference arm does its work on
rank 0 only."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest, job = bench.combine_over_ranks(torch, dist, times[rank], world, torch.device("cpu"))
        out[rank] = (slowest, job)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [31.5, 27.25]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, times, out), nprocs=world, start_method="spawn")
        res = dict(out)
    for r in range(world):
        assert res[r] == (31.5, 31.5 / 2)


def test_single_rank_needs_no_process_group():
    assert bench.combine_over_ranks(torch, None, 12.0, 1, torch.device("cpu")) == (12.0, 12.0)


def test_rank_seeds_are_disjoint():
    """Seeds a rank uses: 4000..4000 + 224 + 10^6 (two G sets), 5000..5224; shifted per rank by
    10^5, more than the span of one rank's seeds inside each family."""
    def seeds(rank):
        off = bench.rank_seed_offset(rank)
        out = set()
        idx = 0
        for (B, _, _) in bench.MEGABATCHES:
            for i in range(B):
                out.add(5000 + idx + i + off)
                for s in range(2):
                    out.add(4000 + idx + i + 10 ** 6 * s + off)
            idx += B
        return out
    a, b = seeds(0), seeds(1)
    assert not (a & b)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "cpu_sample_inputs", lambda *a, **k: called.append(1))

    class Args:
        steps, warmup = 1, 0

    bench.run_reference(Args())
    assert not called
    assert capsys.readouterr().out == ""

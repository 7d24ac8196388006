"""bench.py's multi-rank path on the CPU: two gloo ranks (no GPU).

Each rank reports its own step time; both must agree on the maximum and on
the whole-job throughput (world * step bytes / slowest time), and a reference
run on a non-zero rank must print nothing.
"""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, gbs = bench.aggregate(1.0 + rank, 1_000_000, world, dist)
        out[rank] = (ms, gbs)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_and_job_throughput():
    world = 2
    port = _port()
    with mp.get_context("spawn").Manager() as m:  # no fork of a threaded test process
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for ms, gbs in res.values():
        assert ms == pytest.approx(2.0)
        assert gbs == pytest.approx(world * 1_000_000 / 2.0e-3 / 1e9)


def test_reference_arm_is_silent_on_other_ranks(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        ref_rows = 4
        steps = 1
        warmup = 0

    bench.run_reference(A())
    assert capsys.readouterr().out == ""


def test_single_rank_aggregate_needs_no_process_group():
    assert not dist.is_initialized()
    ms, gbs = bench.aggregate(4.0, 8_000_000, 1)
    assert ms == 4.0 and gbs == pytest.approx(2.0)

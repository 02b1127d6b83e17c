"""The benchmark's multi-rank path on CPU: two gloo ranks (what torchrun
starts on a node, one per GPU) agree on the slowest rank's time, meet at the
barrier, and the whole-job rate counts every rank's keys; the reference arm
runs on rank 0 only.  No GPU is used."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, local, dist = bench.setup_dist(world)
    import torch
    ms = 10.0 + 5.0 * r                       # rank r's (made-up) step time
    slowest = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    bench.barrier(dist)
    out.put((r, w, local, slowest, bench.whole_job_rate(w, 1000, slowest)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert all(x[3] == 15.0 for x in res)           # the slowest rank's time, everywhere
    assert all(x[4] == pytest.approx(2 * 1000 / 15e-3) for x in res)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args) == 0             # rank 1 returns without work or output


def test_whole_job_rate_single_rank():
    assert bench.whole_job_rate(1, 232000, 0.5) == pytest.approx(232000 / 0.5e-3)

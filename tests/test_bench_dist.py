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


def test_packed_inputs_round_trip():
    # the end-to-end step sends its inputs as one buffer: every part's view
    # must hold that input, at an aligned offset, after the single copy
    import torch
    parts = [torch.randn(3, 64, 128).to(torch.bfloat16), torch.randn(3, 64), torch.tensor([5, 7, 9], dtype=torch.int32),
             torch.randn(3, 128).to(torch.bfloat16), torch.tensor([11, 12, 13], dtype=torch.int64)]
    host, dev, views = bench.pack_pinned(parts, "cpu", pin=False)
    dev.zero_()
    dev.copy_(host)
    for t, v in zip(parts, views):
        assert v.dtype == t.dtype and v.shape == t.shape
        assert torch.equal(v, t)
        assert (v.data_ptr() - dev.data_ptr()) % 256 == 0
    assert host.numel() == dev.numel() >= sum(t.numel() * t.element_size() for t in parts)

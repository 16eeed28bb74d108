"""bench.py's host logic on CPU: the multi-rank timing reduction (gloo,
world size 2) and the reference arm's JSON line.

The N > 1 benchmark runs one shard per rank with no data-path collective;
the only cross-rank steps are a barrier and the max of the ranks' times,
which these tests run over gloo on CPU.
"""
import contextlib
import io
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    bench.barrier(world)
    # rank r took (r + 1) * 10 ms per step; the job is as slow as its slowest rank
    t = bench.max_over_ranks(0.010 * (rank + 1), world)
    agg = bench.aggregate(bytes_per_rank=1e9, elems_per_rank=1e8, world=world, seconds=t)
    out[rank] = (t, agg["gbs"], agg["gparams_per_s"])
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank_and_sum_the_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        t, gbs, gps = out[r]
        assert t == pytest.approx(0.020)
        assert gbs == pytest.approx(2 * 1e9 / 0.020 / 1e9)
        assert gps == pytest.approx(2 * 1e8 / 0.020 / 1e9)


def _fits_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    # rank 1 sees a host too small for its pinned gradients
    if rank == 1:
        bench.host_memory_allows = lambda nbytes: False
    out[rank] = bench.e2e_fits(1 << 30, world)
    dist.destroy_process_group()


def test_end_to_end_leg_is_skipped_by_all_ranks_or_none():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_fits_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] is False and out[1] is False


def test_host_memory_check(monkeypatch):
    monkeypatch.setattr(bench.os, "sysconf",
                        lambda name: {"SC_AVPHYS_PAGES": 1000, "SC_PAGE_SIZE": 4096}[name])
    assert bench.host_memory_allows(2_048_000)
    assert not bench.host_memory_allows(2_048_001)
    assert bench.e2e_fits(2_048_000, 1) and not bench.e2e_fits(3_000_000, 1)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.aggregate(28.0, 1.0, 1, 1.0) == {"gbs": 28e-9, "gparams_per_s": 1e-9}


def test_reference_arm_prints_one_json_line(monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3",
                         "--ref-tensors", "1"])
    assert rc == 0
    lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert rc == 0 and buf.getvalue() == ""


def test_warmup_below_three_is_refused():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_kernel_source_hash_is_stable_and_covers_the_sources():
    assert bench.kernel_source_hash() == bench.kernel_source_hash()
    names = {os.path.basename(p) for p in bench.KERNEL_SOURCES}
    assert {"fadam.h", "fadam_kernel.cuh", "fadam_plan.cu"} <= names

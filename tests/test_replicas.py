"""Host logic of the multi-replica benchmark (one process per GPU, no data-path
collective): checked with two gloo processes on the CPU. The job's step time is
the slowest replica's; its throughput counts every replica's tokens; the
reference arm runs on rank 0 only."""
import io
import contextlib
import multiprocessing as mp
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step = bench.max_over_ranks(1.5 + rank, world)   # rank 1 is the slow one
        q.put((rank, step, bench.whole_job_rate(4096, world, step)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_step_and_the_whole_job():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in procs)
    assert [g[1] for g in got] == [2.5, 2.5]
    assert all(abs(g[2] - 2 * 4096 / 2.5e-3) < 1e-6 for g in got)


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_rate(4096, 1, 2.0) == pytest.approx(2048000.0)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.run_reference(types.SimpleNamespace(steps=1, warmup=3), rank=1, world=2)
    assert out.getvalue() == ""


def test_extra_legs_and_dominant_site_selection():
    sys.path.insert(0, ROOT)
    import bench
    args = types.SimpleNamespace(no_extras=False, legs="all")
    assert all(bench.leg_on(args, leg) for leg in bench.EXTRA_LEGS)
    args.legs = "down,decode"
    assert bench.leg_on(args, "down") and bench.leg_on(args, "decode") and not bench.leg_on(args, "hybrid")
    args.no_extras = True
    assert not any(bench.leg_on(args, leg) for leg in bench.EXTRA_LEGS)
    # a site whose kernels overlap another site's (its events span both) is never the dominant one
    times = {1: 83.0, 2: 99.0, 3: 113.0, 4: 117.0, 5: 232.0, 6: 198.0}
    assert 5 in bench.CONCURRENT_SITES and bench.dominant_site(times) == 6

"""The N-GPU path of the benchmark is replicas only: each rank runs its own
workload and the job value is all ranks' work over the slowest rank's time.
Checked here with two gloo ranks on CPU (no GPU, no data-path collective):
the arithmetic alone, and the benchmark's own rank skeleton (process group
from the launcher's environment, warm-up, barriers around the timed region,
max over ranks, teardown) driven by a CPU step."""
import os
import socket
import time

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    seconds = [2.0, 3.0][rank]
    value, slowest = bench.replica_value(seconds, 6e12, world)
    out.put((rank, value, slowest, bench.dist_env()))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_value_takes_max_time_and_sums_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, slowest, env in res:
        assert slowest == 3.0                       # max over ranks
        assert value == pytest.approx(2 * 6e12 / 3.0 / 1e12)
        assert env == (2, rank, rank)


def test_single_process_value():
    import bench
    v, s = bench.replica_value(1.5, 3e12, 1)
    assert s == 1.5 and v == pytest.approx(2.0)


def _cpu_time(step, n):
    """time_launches' contract on the host clock: per-step ms and region ms."""
    t0 = time.perf_counter()
    times = []
    for _ in range(n):
        s = time.perf_counter()
        step()
        times.append((time.perf_counter() - s) * 1e3)
    return times, (time.perf_counter() - t0) * 1e3


def _skeleton_rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.init_replicas()
    calls = []
    # rank 1's steps are slower; rank 0's region must still wait for it at
    # the closing barrier
    step = lambda: (calls.append(1), time.sleep(0.002 if r == 0 else 0.02))
    times, region_ms = bench.replica_region(step, steps=5, warmup=3, world=w,
                                            sync=lambda: None, time_fn=_cpu_time)
    value, slowest = bench.replica_value(region_ms * 1e-3, 1e12, w)
    out.put((r, local, w, len(calls), len(times), region_ms, value, slowest))
    bench.finish_replicas(w)


def test_benchmark_rank_skeleton_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_skeleton_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    regions = [r[5] for r in res]
    for rank, local, world, ncalls, ntimes, region_ms, value, slowest in res:
        assert (local, world) == (rank, 2)
        assert ncalls == 3 + 5 and ntimes == 5          # warm-up untimed, K steps timed
        assert slowest == pytest.approx(max(regions) * 1e-3)
        assert value == pytest.approx(2 * 1e12 / slowest / 1e12)
    assert regions[1] >= 5 * 20 * 0.9                    # the slow rank's own steps

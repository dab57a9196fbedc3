"""The N-GPU path of the benchmark is replicas only: each rank runs its own
workload and the job value is all ranks' work over the slowest rank's time.
Checked here with two gloo ranks on CPU (no GPU, no data-path collective)."""
import os
import socket

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

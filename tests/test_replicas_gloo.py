"""The multi-rank bench logic (replicas, max over ranks) on two gloo ranks (CPU).

bench.py runs one independent replica per GPU under torchrun; the only
cross-rank step is taking the max of the per-rank timings, checked here with
world size 2 on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    assert bench.dist_env() == (world, rank, rank)
    vals = bench.max_over_ranks([1.0 + rank, 10.0 - rank], world, torch.device("cpu"))
    q.put((rank, vals))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [2.0, 10.0]


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks([3.5, 1.0], 1, None) == [3.5, 1.0]

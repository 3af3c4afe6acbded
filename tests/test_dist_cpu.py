"""Host-side multi-process path of bench.py (replicas only: no data-path
collective): two gloo ranks on the CPU agree on the barrier and on the
maximum of their step times."""
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


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    d = bench.dist_init(ws)
    bench.barrier(d)
    results[rank] = bench.reduce_max(1.5 + rank, d)
    bench.barrier(d)
    d.destroy_process_group()


def test_two_gloo_ranks_reduce_max():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    assert dict(results) == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_group():
    import bench
    assert bench.dist_init(1) is None
    assert bench.reduce_max(3.0, None) == 3.0

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


def test_gpus_flag_spawns_or_checks_the_world():
    """--gpus N without torchrun starts N ranks; under torchrun WORLD_SIZE must
    equal N."""
    import bench
    assert bench.check_world(1, environ={}) == "run"
    assert bench.check_world(4, environ={}) == "spawn"
    assert bench.check_world(2, environ={"WORLD_SIZE": "2"}) == "run"
    with pytest.raises(SystemExit):
        bench.check_world(8, environ={"WORLD_SIZE": "1"})
    cmd = bench.launcher_cmd(3, ["--gpus", "3", "--steps", "5"], port=29411)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=3" in cmd and "--master-addr=127.0.0.1" in cmd and "--master-port=29411" in cmd
    assert cmd[-4:] == ["--gpus", "3", "--steps", "5"] and cmd[-5].endswith("bench.py")


def test_gpus_flag_starts_two_gloo_replicas():
    """bench.py --gpus 2 really starts two ranks (gloo on the CPU; the launch
    check does no GPU work) and rank 0 prints one line."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--check-launch"],
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0]) == {"world_size": 2, "rank_sum": 1}


def test_roofline_model_matches_hand_counts():
    """Step bytes of the qwen35moe-shaped layer at 1 token with 8 experts
    selected: 8 x 6.29 MB of expert weights + the 257 x 2048 bf16 router + the
    6.29 MB shared expert + x (bf16) and out (fp32)."""
    import bench
    import synth
    m = bench.Model(synth.QWEN)
    per_expert = 3 * 2048 * 512 * 2
    want = 8 * per_expert + 257 * 2048 * 2 + per_expert + 2048 * (2 + 4)
    assert m.step_bytes(1, 8) == want
    assert m.step_flops(4096) == 2.0 * 4096 * 8 * 3 * 2048 * 512 + 2.0 * 4096 * 3 * 2048 * 512 + 2.0 * 4096 * 2048 * 256
    mx = bench.Model(synth.GPTOSS_MXFP4)
    assert mx.up_per_expert == 2 * 2880 * 2880 * (0.5 + 1 / 32) + 2 * 2880 * 4

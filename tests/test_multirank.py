"""N>1 host logic of bench.py on CPU: two gloo ranks, each timing its own
replica; the job takes the slowest rank's time and counts every rank's units."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [10.0 + 5.0 * rank, 20.0 - 3.0 * rank]
    got = bench.max_over_ranks(mine, dist)
    dist.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [15.0, 20.0]


def test_whole_job_value_counts_every_replica():
    import bench
    one = bench.whole_job_tflops(75.5e9, 10, 1, 5.0)
    two = bench.whole_job_tflops(75.5e9, 10, 2, 5.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(75.5e9 * 10 / 5e-3 / 1e12)
    assert bench.max_over_ranks([1.0, 2.0], None) == [1.0, 2.0]


def test_reference_arm_under_torchrun_prints_once():
    """bench.py --impl reference launched as the N>1 bench is (torchrun, two
    ranks): rank 0 alone times the oracle and prints one JSON line; the other
    rank exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--config", "1", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # the CUDA arm builds its `config` with the same function: the two arms' objects are identical
    import argparse
    sys.path.insert(0, root)
    import bench
    args = argparse.Namespace(config=1, tokens=None)
    assert d["config"] == bench.run_config(bench.workload(1), args, "fwd", 2)

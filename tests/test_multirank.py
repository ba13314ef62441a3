"""The multi-rank path of the bench on CPU (gloo, world size 2).

The grouped GEMM has no exchange step: each rank runs its own replica of the
workload, so the only cross-rank logic is the barrier, the max-over-ranks time
and the whole-job aggregate, and the reference arm's rank-0-only rule.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    slowest = bench.reduce_max(1.5 + rank, world, "cpu")   # rank 1 is the slow one
    out[rank] = (slowest, bench.aggregate_tflops(world, 1e12, slowest))
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_gloo():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5
    assert res[0][1] == pytest.approx(2 * 1e12 / 2.5e-3 / 1e12)


def test_aggregate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_tflops(1, 2e12, 1.0) == pytest.approx(2000.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "2", "--warmup", "3", "--gpus", "2"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "tiny"

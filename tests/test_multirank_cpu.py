"""Multi-rank paths of the benchmark on CPU (gloo, world size 2).

The method has no exchange step, so N GPUs run independent replicas; the only
cross-rank operations are the barrier and the max over ranks of the step
time.  These run here with the gloo backend on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                                         rank=rank, world_size=2)
    try:
        torch.distributed.barrier()
        out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank)
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(free_port(), out), nprocs=2, join=True)
    assert out[0] == 15.0 and out[1] == 15.0


def test_max_over_ranks_without_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference under torchrun: rank 0 prints one JSON line,
    the other rank exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--ref-rows", "8"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0

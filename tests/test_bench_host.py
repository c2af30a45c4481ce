"""CPU tests of bench.py's host logic: byte/flop accounting, the reference
(oracle) arm, and the multi-rank reductions under torchrun with gloo."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_decode_bytes_accounting():
    # L=100: all BF16 (100 tokens * 1152); L=1000: 132 BF16 + 868 packed
    assert bench.decode_bytes([100], "C4R4", 1, 16) == 100 * 1152 + 16 * (1152 + 1024 + 4)
    assert bench.decode_bytes([1000], "C4R4", 1, 16) == 132 * 1152 + 868 * 324 + 16 * 2180
    assert bench.decode_bytes([1000], "C2R4", 1, 16) == 132 * 1152 + 868 * 196 + 16 * 2180
    assert bench.decode_bytes([1000], "BF16", 1, 16) == 1000 * 1152 + 16 * 2180
    assert bench.decode_flops([10, 20], 16) == 30 * 2 * 16 * 1088


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_reference_arm_single_process():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--ref-budget", "0.05", "--workload", "tiny_c4r4"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["unit"] == "GB/s"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-budget", "0.05",
           "--workload", "tiny_c4r4"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout  # rank 0 only
    assert json.loads(lines[0])["n_gpus"] == 2


def _reduce_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mx = bench.max_over_ranks(float(rank + 1), world, "cpu")
    sm = bench.sum_over_ranks(float(rank + 1), world, "cpu")
    bench.barrier(world)
    dist.destroy_process_group()
    q.put((rank, mx, sm))


def test_rank_reductions_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_reduce_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, mx, sm in res:
        assert mx == 2.0 and sm == 3.0

"""The N > 1 path of bench.py on the host, with world size 2 over gloo.

Decode does not shard here: bench.py --gpus N runs N independent replicas,
one per rank, joined only by a barrier and a max over the ranks' times, and
rank 0 alone prints the line.  These tests run that plumbing as two CPU
processes (no GPU is touched: CUDA is hidden from the children)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world), "CUDA_VISIBLE_DEVICES": ""})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank's time differs; every rank must get the slowest one
    m = bench.max_over_ranks(1.5 + rank, w)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(m))
    bench.barrier(w)
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_world_size_two(tmp_path):
    port = free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(2)]
    assert got == [2.5, 2.5]


def test_reference_arm_under_torchrun_prints_one_line(tmp_path):
    """torchrun with two ranks: rank 0 times the oracle and prints the one
    JSON line; the other rank exits 0 without work."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--workload", "tiny",
           "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0

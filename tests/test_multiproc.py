"""Multi-process host logic of the benchmark (replicas, no data-path
collective) on CPU with the gloo backend, world size 2."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local, d = bench.dist_setup(world)
    assert (r, w) == (rank, world) and d is dist
    bench.barrier(d)
    m = bench.max_over_ranks(d, float(rank + 1) * 1.5)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "max": m}, f)
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path, monkeypatch):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    # CPU ranks: no GPU is visible to them, also where one is present
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "")
    mp.start_processes(_worker, args=(2, free_port(), str(tmp_path)), nprocs=2, start_method="spawn")
    for rank in range(2):
        d = json.load(open(tmp_path / f"rank{rank}.json"))
        assert d["max"] == 3.0
    del torch


def test_reference_arm_under_torchrun():
    """Under torchrun only rank 0 runs and prints the reference line; the
    other rank exits 0 without work."""
    pytest.importorskip("torch")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "4", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")  # CPU ranks, also on a GPU machine
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "us/call"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0

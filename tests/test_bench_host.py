"""Host-side logic of bench.py on the CPU: the max-over-ranks reduction of
the replica timing across two gloo processes, and the reference arm (the
oracle on the host cores) under torchrun with two ranks, where rank 0 alone
prints the JSON line.  No GPU is used."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    out[rank] = bench._reduce_max(1.5 + rank, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_time_is_the_max_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_reduce_max_without_a_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._reduce_max(3.25, torch.device("cpu")) == 3.25


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched as the driver launches it for
    N > 1: rank 0 times the oracle and prints one JSON line; rank 1 exits 0
    without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0

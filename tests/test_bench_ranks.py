"""The multi-process side of bench.py on the CPU: world size 2 over gloo.

A multi-GPU run is replicas only (each rank its own workload and pools, no
data-path exchange), so what there is to test without GPUs is the host
logic: the ranks line up at a barrier, a per-rank figure is reduced to its
maximum over the ranks, only rank 0 reports, and the reference arm launched
under torchrun prints one line from rank 0 while the other rank exits
cleanly.  Rendezvous on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r = bench.Ranks(dist, torch.device("cpu"))
        r.barrier()
        got = r.max([rank + 1.0, 10.0 - rank, -float(rank), 0.25 * (rank + 1)])
        r.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"rank": r.rank, "world": r.world, "main": r.main, "max": got}, f)
    finally:
        dist.destroy_process_group()


def test_ranks_single_process_is_local():
    r = bench.Ranks()
    assert (r.rank, r.world, r.main) == (0, 1, True)
    r.barrier()
    assert r.max([1.5, -2, 3]) == [1.5, -2.0, 3.0]


def test_ranks_max_and_barrier_over_gloo(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == world
        assert d["main"] == (r == 0)
        # every rank gets the maximum over both ranks, element by element
        assert d["max"] == [2.0, 10.0, 0.0, 0.5]


def test_reference_arm_under_torchrun_reports_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 1 and d["value"] > 0

"""Multi-process host logic of the replicas-only benchmark, on CPU.

The path shards with no exchange, so `bench.py --gpus N` runs N independent
replicas; what spans the ranks is host logic only: the process group set-up,
the max-over-ranks reduction of the timed region, and the reference arm, which
rank 0 alone runs.  These run as gloo ranks (world size 2) on the CPU.
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


def _rank_main(rank, world, port, values, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), TCL_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    r, w, dist = bench.dist_setup(world)
    assert (r, w) == (rank, world) and dist is not None
    got = bench.max_over_ranks(values[rank], dist)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "max": got}, f)


def test_max_over_ranks_gloo(tmp_path):
    values = [3.25, 7.5]  # rank 1 is the slower one
    mp.spawn(_rank_main, args=(2, _free_port(), values, str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        d = json.load(open(tmp_path / f"rank{rank}.json"))
        assert d == {"rank": rank, "world": 2, "max": max(values)}


def test_single_rank_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.delenv("RANK", raising=False)
    assert bench.dist_setup(1) == (0, 1, None)
    assert bench.dist_setup(4) == (0, 1, None)  # launched without torchrun
    assert bench.max_over_ranks(1.5, None) == 1.5


def test_reference_arm_under_torchrun():
    """Two ranks, one JSON line (rank 0's), both ranks exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "3", "--warmup", "3", "--config", "distinct", "--ref-seconds", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}

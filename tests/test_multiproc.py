"""The multi-replica host path of bench.py on CPU: two processes on a gloo group.

A benchmark with N > 1 runs N independent replicas (the method shards by block range, and
one GPU holds every stage, so there is no data-path collective): ranks come from the
launcher's environment, the timed duration is the maximum over ranks, the value is the
units of all ranks over that duration, and only rank 0 prints.  The GPU part of a replica
is the single-GPU path tested elsewhere.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    m = bench.max_over_ranks(1.5 + r, dist)  # rank 1 is the slow replica
    rate = bench.aggregate_rate(64, m, w)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "max": m, "rate": rate}, f)


def test_max_over_ranks_and_aggregate_on_gloo(tmp_path):
    port = free_port()
    torch.multiprocessing.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                                          start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [x["rank"] for x in res] == [0, 1] and all(x["world"] == 2 for x in res)
    assert all(x["max"] == 2.5 for x in res)                 # the slowest rank's time
    assert all(abs(x["rate"] - 64 * 2 / 2.5) < 1e-12 for x in res)  # units of both ranks / that time


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as 2 ranks: rank 0 runs the oracle and prints one
    JSON line, rank 1 leaves without work."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--cpu-budget", "0.1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["metric"] == "decode tok/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0

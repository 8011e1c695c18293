"""The N > 1 launch contract on the CPU (gloo, world size 2): the benchmark
runs one replica per rank with no collective on the data path (the FFN
shards by token with no exchange), and its only cross-rank step is the
timing reduction, the maximum over ranks, which every rank receives.  The
reference arm under torchrun prints exactly one JSON line, from rank 0."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = 10.0 * (rank + 1) + 0.25  # rank 1 is the slower replica
        got = bench.max_over_ranks(torch, mine, world, torch.device("cpu"))
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_timing_reduction_is_the_max_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    got = [float(open(tmp_path / f"r{r}.txt").read()) for r in range(2)]
    assert got == [20.25, 20.25]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(torch, 3.5, 1, torch.device("cpu")) == 3.5


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_once(tmp_path):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=560)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"

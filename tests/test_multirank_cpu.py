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


# ---- token-sharded training step: ranges and the weight-gradient sum -------

def test_token_ranges_cover_every_token_once():
    from activation_sparse_transformer_gate_gb300 import shard
    for T in (1, 127, 128, 129, 1000, 4096, 4097):
        for world in (1, 2, 3, 4, 8):
            rs = [shard.token_range(T, r, world) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == T
            for (a0, a1), (b0, b1) in zip(rs, rs[1:]):
                assert a1 == b0 and a0 <= a1
            for r, (a0, a1) in enumerate(rs):   # whole 128-token blocks except the tail
                assert (a0 % 128 == 0 or a0 == T) and (a1 % 128 == 0 or a1 == T)
            sizes = [(a1 - a0 + 127) // 128 for a0, a1 in rs]
            assert max(sizes) - min(sizes) <= 1 or T < 128 * world


def _shard_main(rank, world, port, out_dir):
    """Each rank: the oracle's backward on its token range (standing in for
    the library's per-rank backward, which needs a GPU), then the
    all-reduce of the weight gradients."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import numpy as np
        import oracle
        import synth
        from activation_sparse_transformer_gate_gb300 import shard
        w = synth.Workload("sh", 300, 64, 256, 64, 4, "bf16", True, -1.5, 77, hot_tokens=2,
                           seq_len=100, hot_bias=1.4, lam=1e-3, train=True)
        a = synth.generate(w)
        t0, t1 = shard.token_range(w.T, rank, world)
        sl = slice(t0, t1)
        rb = None if a["rb"] is None else a["rb"][sl]
        b = oracle.ffn_backward(a["x"][sl], a["Wg"], a["bg"], rb, a["Wu"], a["Wd"], a["dy"][sl],
                                w.lam, "bf16", "bf16")
        grads = [torch.from_numpy(np.ascontiguousarray(b[k])) for k in ("dWg", "dWu", "dWd", "dbg")]
        shard.allreduce_weight_grads(grads)
        np.savez(os.path.join(out_dir, f"g{rank}.npz"), *[g.numpy() for g in grads],
                 dx=b["dx"], t0=t0, t1=t1)
    finally:
        dist.destroy_process_group()


def test_token_sharded_backward_sums_to_the_whole_batch(tmp_path):
    import numpy as np
    import oracle
    import synth
    port = _free_port()
    mp.start_processes(_shard_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    w = synth.Workload("sh", 300, 64, 256, 64, 4, "bf16", True, -1.5, 77, hot_tokens=2,
                       seq_len=100, hot_bias=1.4, lam=1e-3, train=True)
    a = synth.generate(w)
    full = oracle.ffn_backward(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], a["dy"],
                               w.lam, "bf16", "bf16")
    parts = [np.load(tmp_path / f"g{r}.npz") for r in range(2)]
    assert int(parts[0]["t0"]) == 0 and int(parts[0]["t1"]) == int(parts[1]["t0"])
    assert int(parts[1]["t1"]) == w.T
    for i, k in enumerate(("dWg", "dWu", "dWd", "dbg")):
        for p in parts:                      # every rank holds the batch's sum
            got, ref = p[f"arr_{i}"], full[k]
            assert np.max(np.abs(got - ref)) <= 1e-9 * max(np.max(np.abs(ref)), 1.0), k
    dx = np.concatenate([p["dx"] for p in parts])   # dx needs no exchange
    assert np.array_equal(dx, full["dx"])

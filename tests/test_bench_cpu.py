"""Host logic of bench.py's per-kernel rooflines (no GPU): which kernels
are rated against which roofline, and the algorithmic work of each, for the
dispatcher's two dh paths."""
import numpy as np

import bench
import synth


def kern_times(names, ms=0.1):
    return {n: {"avg_ms": ms, "ms_per_step": ms, "launches_per_step": 1.0} for n in names}


def small_case():
    w = synth.Workload("bc", 256, 128, 512, 128, 8, "bf16", True, -2.33, 5, lam=1e-4, train=True)
    rng = np.random.default_rng(5)
    nnz = rng.integers(0, 4, size=(w.F // w.C, w.T))  # no row overflows (K = 8)
    return w, nnz


def test_dh_sddmm_is_rated_on_bytes():
    w, nnz = small_case()
    names = ["bwd_slots_sddmm", "bwd_dh_gemm_sampled", "gate_gemm_relu_twell"]
    rl = bench.kernel_rooflines(kern_times(names), w, nnz, True, 0, 0, dh_gemm=False)
    a = int(nnz.sum())
    r = rl["bwd_slots_sddmm"]
    assert r["bound"] == "hbm" and r["algorithmic"] == a * (w.D * 2 + 14) + w.T * w.D * 2
    assert "bwd_dh_gemm_sampled" not in rl  # launched but idle: not rated
    assert rl["gate_gemm_relu_twell"]["algorithmic"] == 2.0 * w.T * w.D * w.F


def test_dh_gemm_is_rated_on_flops_of_the_whole_product():
    w, nnz = small_case()
    names = ["bwd_slots_sddmm", "bwd_dh_gemm_sampled"]
    rl = bench.kernel_rooflines(kern_times(names, 0.05), w, nnz, True, 0, 0, dh_gemm=True)
    r = rl["bwd_dh_gemm_sampled"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["algorithmic"] == 2.0 * w.T * w.D * w.F
    assert abs(r["achieved"] - 2.0 * w.T * w.D * w.F / 0.05e-3 / 1e12) < 1e-9
    assert "bwd_slots_sddmm" not in rl  # launched but idle: not rated

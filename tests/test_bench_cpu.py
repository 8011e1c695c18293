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


def test_dh_gemm_also_rated_on_the_sddmm_bytes():
    w, nnz = small_case()
    rl = bench.kernel_rooflines(kern_times(["bwd_dh_gemm_sampled"], 0.05), w, nnz, True, 0, 0,
                                dh_gemm=True)
    r = rl["bwd_dh_gemm_sampled"]
    a = int(nnz.sum())
    assert r["sddmm_bytes"] == a * (w.D * 2 + 14) + w.T * w.D * 2
    assert abs(r["sddmm_equivalent_gbs"] - r["sddmm_bytes"] / 0.05e-3 / 1e9) < 1e-6


def test_gather_dominated_step_is_read_against_the_l2_gather_rate():
    """An L2-served gather kernel: bound "l2" against the measured gather
    rate (frac <= 1 when below it), with its HBM figures beside it."""
    w, nnz = small_case()
    kern = kern_times(["bwd_dw_gather", "gate_gemm_relu_twell"], 0.01)
    kern["bwd_dw_gather"]["ms_per_step"] = 0.2
    rl = bench.kernel_rooflines(kern, w, nnz, True, 0, 0)
    alg = rl["bwd_dw_gather"]["achieved"]
    r = bench.dominant_roofline(kern, rl, "c2", True, gceil=2 * alg)
    assert r["kernel"] == "bwd_dw_gather" and r["bound"] == "l2"
    assert abs(r["frac"] - 0.5) < 1e-3 and r["unit"] == "GB/s"
    assert r["hbm"]["frac_algorithmic_bytes"] == round(rl["bwd_dw_gather"]["frac"], 4)
    # without a measured gather rate the HBM reading is kept
    r2 = bench.dominant_roofline(kern, rl, "c2", True, gceil=None)
    assert r2["bound"] == "hbm"


def test_fp32_gate_gemm_is_rated_on_the_alu_peak():
    w = synth.scaled(synth.config1(), train=False)
    nnz = np.zeros((w.F // w.C, w.T), dtype=np.int64)
    nnz[0, :] = 1
    rl = bench.kernel_rooflines(kern_times(["gate_gemm_relu_twell", "twell_updown_fused"]), w,
                                nnz, False)
    assert rl["gate_gemm_relu_twell"]["bound"] == "alu"
    assert abs(rl["gate_gemm_relu_twell"]["peak"] - bench.fp32_alu_tflops()) < 1e-9
    # fp32 rows: 4-byte elements, one gathered weight row per pair (plain FFN)
    pairs = int(nnz.sum())
    twell = (w.F // w.C) * w.T * (5 * w.K + 1)
    want = pairs * w.D * 4 + w.T * w.D * 4 + twell
    assert rl["twell_updown_fused"]["algorithmic"] == want


def test_dw_gather_is_read_against_its_own_rows_probe():
    """Per-kernel ceilings: the weight-gradient gather (token rows of x and
    dy) is rated on the token-row probe, the others on the weight-row one."""
    w, nnz = small_case()
    kern = kern_times(["bwd_dw_gather", "bwd_dx_spmm"], 0.01)
    kern["bwd_dw_gather"]["ms_per_step"] = 0.2
    rl = bench.kernel_rooflines(kern, w, nnz, True, 0, 0)
    alg = rl["bwd_dw_gather"]["achieved"]
    ceil = {"bwd_dw_gather": 4 * alg, "bwd_dx_spmm": 2 * alg,
            "_source": {"bwd_dw_gather": "token rows"}}
    r = bench.dominant_roofline(kern, rl, "c2", True, ceil)
    assert r["kernel"] == "bwd_dw_gather" and abs(r["frac"] - 0.25) < 1e-3
    assert "token rows" in r["peak_source"]

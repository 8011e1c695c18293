"""GPU parity of the sparse backward (per-token SDDMM + dx SpMM, sparse
transpose, dW gathers, overflow rows from the dense backup, L1 term) against
the CPU oracle."""
import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import oracle
import synth
from twell_testlib import check_backward, ctl_fields, dh_gemm_of, run_train

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    tw.load()


def test_bf16_gated_small_with_overflow_rows():
    w = synth.Workload("bw", 300, 256, 1024, 128, 8, "bf16", True, -2.33, 21, hot_tokens=3,
                       seq_len=100, hot_bias=1.49, train=True)
    a = synth.generate(w)
    g = run_train(a, w, 1e-4)
    assert g["code"] == 0 and g["n_ovf"] >= 9
    check_backward(a, w, g, 1e-4)


def test_l1_term_dominant():
    """lambda comparable to dy . Wd: the L1 gradient matters in every entry."""
    w = synth.Workload("l1", 160, 256, 512, 64, 8, "bf16", True, -1.8, 22, train=True)
    a = synth.generate(w)
    g = run_train(a, w, 0.5)
    assert g["code"] == 0
    check_backward(a, w, g, 0.5)


def test_zero_down_weight_closed_form():
    """W_down = 0: y = 0 and dbg[n] = lambda * sum over active tokens of |u|."""
    w = synth.Workload("wd0", 128, 256, 512, 128, 8, "bf16", True, -1.5, 23, train=True)
    a = synth.generate(w)
    a["Wd"] = np.zeros_like(a["Wd"])
    g = run_train(a, w, 0.25)
    assert g["code"] == 0
    assert np.all(g["y"] == 0)
    b = check_backward(a, w, g, 0.25)
    assert np.abs(b["dbg"]).max() > 0


def test_config1_fp32_nongated():
    w = synth.scaled(synth.config1(), train=True)
    a = synth.generate(w)
    g = run_train(a, w, 1e-3)
    assert g["code"] == 0
    check_backward(a, w, g, 1e-3)


def test_nongated_bf16_with_overflow():
    w = synth.Workload("ngb", 200, 256, 512, 64, 4, "bf16", False, -1.7, 24, hot_tokens=2,
                       seq_len=50, hot_bias=1.5, train=True)
    a = synth.generate(w)
    g = run_train(a, w, 0.05)
    assert g["code"] == 0 and g["n_ovf"] >= 8
    check_backward(a, w, g, 0.05)


def test_many_overflow_rows_dense_gemm_path():
    """>= 128 overflow rows (but fewer than half): forward and backward run them
    on the tensor-core dense-row GEMMs (a partial last tile of rows, so the
    weight-gradient GEMMs contract over zero-padded rows); the other rows take
    the gather kernels, and the two weight-gradient parts add up."""
    w = synth.Workload("bmany", 600, 256, 1024, 128, 8, "bf16", True, -2.33, 26, hot_tokens=2,
                       seq_len=7, hot_bias=1.6, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, 1e-3, out=out)
    assert g["code"] == 0 and 128 <= g["n_ovf"] < 300 and g["n_ovf"] % 64 != 0
    n_rows, dense, n_ovf, ovf_gemm = ctl_fields(out["ctl_bwd"])
    assert (dense, ovf_gemm, n_rows) == (0, 1, n_ovf) and n_ovf == g["n_ovf"]
    check_backward(a, w, g, 1e-3)


def test_transpose_several_token_chunks_ragged():
    """T = 2500: the sparse transpose runs over three chunks of 1024 tokens, the
    last one partial, so every list spans chunk boundaries."""
    w = synth.Workload("bchunk", 2500, 256, 512, 128, 8, "bf16", True, -1.2, 27, hot_tokens=2,
                       seq_len=500, hot_bias=1.5, train=True)
    a = synth.generate(w)
    g = run_train(a, w, 1e-3)
    assert g["code"] == 0 and g["n_ovf"] >= 1
    check_backward(a, w, g, 1e-3)


def test_backward_after_density_switched_dense_forward():
    """~5% active, K = 16: forward and backward run every row densely (density
    test on; the backward rebuilds the g / u rows from the slots)."""
    w = synth.Workload("bdens", 160, 256, 1024, 128, 16, "bf16", True, -1.64, 44, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, 1e-3, dense_density=0.0, out=out)
    assert g["code"] == 0
    assert ctl_fields(out["ctl"])[1] == 1  # the forward ran densely
    assert ctl_fields(out["ctl_bwd"])[:2] == (160, 1)  # and so did the backward
    check_backward(a, w, g, 1e-3)


@pytest.mark.parametrize("gated", [True, False])
def test_dense_backward_all_rows_ragged(gated):
    """Every row on the tensor-core backward (density test forced), with
    overflow rows (g / u from the dense backup rows) among rows rebuilt from
    their slots; T = 300 (a partial tile of rows) and d_model 200 (partial
    K block and partial output columns in dx and dW)."""
    w = synth.Workload(f"bdr{int(gated)}", 300, 200, 1024, 128, 8, "bf16", gated, -2.0, 45,
                       hot_tokens=3, seq_len=100, hot_bias=1.4, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, 0.05, dense_density=1e-6, out=out)
    assert g["code"] == 0 and g["n_ovf"] >= 3
    assert ctl_fields(out["ctl_bwd"])[:2] == (300, 1)
    check_backward(a, w, g, 0.05)


def test_fp32_dense_forward_then_gather_backward():
    """fp32 (no tensor-core path): a forward that the density test runs
    densely on the CUDA-core GEMMs (u at the slots filled from its u rows),
    then the gather backward over every row."""
    w = synth.Workload("bf32dense", 96, 256, 512, 64, 8, "f32", True, -1.64, 52, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, 1e-3, dense_density=1e-6, out=out)
    assert g["code"] == 0
    assert ctl_fields(out["ctl"])[1] == 1       # the forward ran densely
    assert ctl_fields(out["ctl_bwd"])[:2] == (0, 0)  # the backward gathered
    check_backward(a, w, g, 1e-3)


def test_dense_backward_l1_and_zero_down_weight():
    """All-dense backward with W_down = 0: dh is the L1 term alone, so
    dbg[n] = lambda * sum over active tokens of |u| (gated) exactly as on
    the gather path."""
    w = synth.Workload("bdwd0", 256, 256, 512, 64, 8, "bf16", True, -1.5, 46, train=True)
    a = synth.generate(w)
    a["Wd"] = np.zeros_like(a["Wd"])
    out = {}
    g = run_train(a, w, 0.25, dense_density=1e-6, out=out)
    assert g["code"] == 0 and ctl_fields(out["ctl_bwd"])[1] == 1
    b = check_backward(a, w, g, 0.25)
    assert np.abs(b["dbg"]).max() > 0


def test_dense_regime_sampled():
    """A dense regime at scale (5% active, K = 16, T = 2048, d_model 1024,
    d_ff 4096): the dispatcher's default density test sends forward and
    backward to the tensor cores; sampled tokens and neurons against the
    oracle."""
    w = synth.Workload("bdreg", 2048, 1024, 4096, 128, 16, "bf16", True, -1.64, 47, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, 1e-4, dense_density=0.0, out=out)
    assert g["code"] == 0 and ctl_fields(out["ctl_bwd"])[:2] == (2048, 1)
    rng = np.random.default_rng(47)
    ts = np.unique(np.concatenate([np.arange(4), rng.choice(w.T, 20, replace=False)]))
    ns = np.unique(np.concatenate([np.arange(4), rng.choice(w.F, 20, replace=False)]))
    check_backward(a, w, g, 1e-4, tok_sel=ts, neu_sel=ns)


@pytest.mark.parametrize("D", [512, 1024])
def test_bf16_dmodel_shapes(D):
    """d_model 512 and 1024: the tensor-core dh SDDMM with 2 and 4 chunks per
    warp, and the generic two-vector dx / dW paths."""
    w = synth.Workload(f"bdm{D}", 160, D, 512, 128, 8, "bf16", True, -1.9, 40 + D // 512,
                       hot_tokens=2, seq_len=80, hot_bias=1.5, train=True)
    a = synth.generate(w)
    g = run_train(a, w, 1e-3)
    assert g["code"] == 0 and g["n_ovf"] >= 1
    check_backward(a, w, g, 1e-3)


@pytest.mark.parametrize("dt,D,dense", [("bf16", 8192, False), ("bf16", 8192, True),
                                          ("f32", 4096, False)])
def test_maximum_dmodel(dt, D, dense):
    """The largest d_model the ABI accepts (16 KB rows), on the gather path
    and (bf16) on the tensor-core path of every row, ragged token count."""
    w = synth.Workload(f"bdmax{dt}", 70, D, 256, 64, 4, dt, True, -1.6, 49, hot_tokens=2,
                       seq_len=35, hot_bias=1.5, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, 1e-3, dense_density=1e-6 if dense else -1.0, out=out)
    assert g["code"] == 0 and g["n_ovf"] >= 2
    if dense:
        assert ctl_fields(out["ctl_bwd"])[:2] == (70, 1)
    check_backward(a, w, g, 1e-3)


@pytest.mark.parametrize("shift", [0, 8])
def test_dh_row_loads_aligned_and_16_byte_aligned(shift):
    """The tensor-core dh SDDMM reads W_down rows with 256-bit loads when W_down
    is 32-byte aligned and with 128-bit loads otherwise (the ABI promises 16
    bytes): both give the oracle's gradients."""
    w = synth.Workload(f"bal{shift}", 200, 1024, 512, 128, 8, "bf16", True, -1.9, 50,
                       hot_tokens=2, seq_len=100, hot_bias=1.5, train=True)
    a = synth.generate(w)
    g = run_train(a, w, 1e-3, wd_shift=shift)
    assert g["code"] == 0
    check_backward(a, w, g, 1e-3)


def test_fp32_dmodel1024_exact_shapes():
    """fp32 d_model 1024: 256 vectors per row, the exact-shape dx and dW paths."""
    w = synth.Workload("bf32d1k", 96, 1024, 256, 64, 4, "f32", True, -1.7, 43, train=True)
    a = synth.generate(w)
    g = run_train(a, w, 1e-3)
    assert g["code"] == 0
    check_backward(a, w, g, 1e-3)


@pytest.mark.parametrize("C,K", [(32, 2), (64, 16), (128, 32)])
def test_tile_shapes(C, K):
    w = synth.Workload(f"bt{C}{K}", 96, 128, 512, C, K, "bf16", True, -1.9, 25 + K, train=True)
    a = synth.generate(w)
    g = run_train(a, w, 1e-2)
    assert g["code"] == 0
    check_backward(a, w, g, 1e-2)


def test_config5_full_size_sampled():
    w = synth.config5()
    a = synth.generate(w)
    g = run_train(a, w, w.lam)
    assert g["code"] == 0
    rng = np.random.default_rng(5)
    ts = np.unique(np.concatenate([np.arange(8), rng.choice(w.T, 24, replace=False)]))
    ns = np.unique(np.concatenate([np.arange(8), rng.choice(w.F, 24, replace=False)]))
    check_backward(a, w, g, w.lam, tok_sel=ts, neu_sel=ns)
    assert np.isfinite(g["dWg"]).all() and np.isfinite(g["dx"]).all()


# ---- dh from the tensor-core GEMM read at the slots ------------------------
# The same workloads as above with dh taken from dy W_down^T over every row
# (dh_density tiny): the slots of ordinary rows, every column of overflow
# rows with a backup row, overflow rows on the dense-row GEMMs skipped, the
# sparse transpose's column counts, pad slots, ragged T and d_ff.
DH_GEMM_CASES = {
    "overflow_rows": (dict(T=300, D=256, F=1024, C=128, K=8, gated=True, bg=-2.33, seed=21,
                           hot_tokens=3, seq_len=100, hot_bias=1.49), 1e-4),
    "nongated_c64_k4": (dict(T=200, D=256, F=512, C=64, K=4, gated=False, bg=-2.2, seed=62,
                             hot_tokens=2, seq_len=50, hot_bias=1.5), 0.05),
    "many_overflow_rows": (dict(T=600, D=256, F=1024, C=128, K=8, gated=True, bg=-2.33, seed=63,
                                hot_tokens=2, seq_len=7, hot_bias=1.6), 1e-3),
    "c32_k2": (dict(T=192, D=128, F=512, C=32, K=2, gated=True, bg=-2.6, seed=64), 1e-2),
    "nongated_c128_k8": (dict(T=260, D=256, F=768, C=128, K=8, gated=False, bg=-2.2, seed=71,
                              hot_tokens=2, seq_len=65, hot_bias=1.5), 0.05),
    "c128_k32": (dict(T=96, D=128, F=512, C=128, K=32, gated=True, bg=-1.9, seed=65), 1e-2),
    "dff_384_ragged": (dict(T=333, D=192, F=384, C=128, K=8, gated=True, bg=-1.8, seed=66,
                            hot_tokens=2, seq_len=111, hot_bias=1.5), 1e-3),
    "l1_dominant": (dict(T=160, D=256, F=512, C=64, K=8, gated=True, bg=-1.8, seed=67), 0.5),
    "token_chunks": (dict(T=2500, D=256, F=512, C=128, K=8, gated=True, bg=-2.0, seed=68,
                          hot_tokens=2, seq_len=500, hot_bias=1.5), 1e-3),
}


@pytest.mark.parametrize("case", sorted(DH_GEMM_CASES))
def test_dh_gemm_read_at_slots(case):
    kw, lam = DH_GEMM_CASES[case]
    extra = {k: kw[k] for k in ("hot_tokens", "seq_len", "hot_bias") if k in kw}
    w = synth.Workload(f"dhg_{case}", kw["T"], kw["D"], kw["F"], kw["C"], kw["K"], "bf16",
                       kw["gated"], kw["bg"], kw["seed"], train=True, **extra)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, lam, out=out, dh_density=1e-9)
    assert g["code"] == 0
    n_rows, dense, n_ovf, ovf_gemm = ctl_fields(out["ctl_bwd"])
    assert dense == 0 and dh_gemm_of(out["ctl_bwd"]) == 1
    if case == "many_overflow_rows":
        assert ovf_gemm == 1 and n_rows == n_ovf >= 128
    elif "hot_tokens" in kw:
        assert ovf_gemm == 0 and n_ovf >= 1
    check_backward(a, w, g, lam)


def test_dh_gemm_equals_gathers_on_the_same_inputs():
    """The two dh paths give the same gradients up to fp32 summation order."""
    kw, lam = DH_GEMM_CASES["overflow_rows"]
    w = synth.Workload("dhg_eq", kw["T"], kw["D"], kw["F"], kw["C"], kw["K"], "bf16", True,
                       kw["bg"], kw["seed"], hot_tokens=3, seq_len=100, hot_bias=1.49, train=True)
    a = synth.generate(w)
    o1, o2 = {}, {}
    g1 = run_train(a, w, lam, out=o1, dh_density=-1.0)
    g2 = run_train(a, w, lam, out=o2, dh_density=1e-9)
    assert dh_gemm_of(o1["ctl_bwd"]) == 0 and dh_gemm_of(o2["ctl_bwd"]) == 1
    for k in ("dx", "dWg", "dWu", "dWd", "dbg"):
        ref = g1[k]
        scale = max(float(np.sqrt(np.mean(ref ** 2))), 1e-30)
        assert np.max(np.abs(g2[k] - ref)) <= 2e-2 * scale, k


def test_dh_gemm_not_taken_when_all_dense():
    """An all-dense backward keeps dh on the dense-row GEMM."""
    w = synth.Workload("dhg_dense", 160, 256, 1024, 128, 16, "bf16", True, -1.64, 69, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, 1e-3, dense_density=1e-6, out=out, dh_density=1e-9)
    assert g["code"] == 0 and ctl_fields(out["ctl_bwd"])[:2] == (160, 1)
    assert dh_gemm_of(out["ctl_bwd"]) == 0
    check_backward(a, w, g, 1e-3)


def test_dh_gemm_below_threshold_gathers():
    """A dh_density above the slot density leaves dh on the gather SDDMM."""
    w = synth.Workload("dhg_thr", 160, 256, 512, 128, 8, "bf16", True, -2.33, 70, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, 1e-3, out=out, dh_density=0.5)
    assert g["code"] == 0 and dh_gemm_of(out["ctl_bwd"]) == 0
    check_backward(a, w, g, 1e-3)


def test_config5_full_size_default_dispatcher():
    """The training-step workload at full size with the dispatcher's default
    choice for dh (about 1% active: the tensor-core GEMM read at the slots)."""
    w = synth.config5()
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, w.lam, out=out, dh_density=0.0)
    assert g["code"] == 0 and dh_gemm_of(out["ctl_bwd"]) == 1
    rng = np.random.default_rng(55)
    ts = np.unique(np.concatenate([np.arange(8), rng.choice(w.T, 24, replace=False)]))
    ns = np.unique(np.concatenate([np.arange(8), rng.choice(w.F, 24, replace=False)]))
    check_backward(a, w, g, w.lam, tok_sel=ts, neu_sel=ns)
    assert np.isfinite(g["dWg"]).all() and np.isfinite(g["dx"]).all()


@pytest.mark.parametrize("dh_density", [1e-9, -1.0], ids=["dh_gemm", "dh_sddmm"])
def test_dense_forward_then_sparse_backward_bf16(dh_density):
    """~1.4% active with the dispatcher's default thresholds (forward 1.3%,
    backward 1.56% when the weights fit in L2): the forward runs every row
    densely (its up GEMM writes u at the slots) while the backward gathers
    and reads that u."""
    w = synth.Workload("dfsb", 256, 256, 1024, 128, 8, "bf16", True, -2.2, 72, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, 1e-3, dense_density=0.0, out=out, dh_density=dh_density)
    assert g["code"] == 0
    assert ctl_fields(out["ctl"])[1] == 1       # the forward ran densely
    assert ctl_fields(out["ctl_bwd"])[:2] == (0, 0)  # the backward gathered
    assert dh_gemm_of(out["ctl_bwd"]) == (1 if dh_density > 0 else 0)
    check_backward(a, w, g, 1e-3)

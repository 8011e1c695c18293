"""GPU parity of the forward path (pack, hybrid split, fused up/down, dense
fallback) against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import oracle
import synth
from twell_testlib import (TOL, assert_close_rms, compare_twell, row_ovf_from_nnz, to_np64,
                           torch_dev, value_allowance, z_band)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    tw.load()


def run_forward(a, w, train=False, ovf_cap=None, dense_switch=0.0, D=None, dense_density=-1.0):
    """Forward through the C ABI.  dense_density < 0 keeps the dispatcher's
    density test off (moderately dense test workloads still take the gather
    kernels); the workspace's control block is returned as "ctl"."""
    T, F, C, K = a["x"].shape[0], a["Wg"].shape[0], w.C, w.K
    D = a["x"].shape[1]
    dtype = tw.TWELL_BF16 if w.dtype == "bf16" else tw.TWELL_F32
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dev = {k: torch_dev(a[k]) for k in ("x", "Wg", "Wu", "Wd", "bg", "rb")}
    bufs = tw.TwellBuffers(T, F, C, K, dtype, ovf_cap, train, dense_switch=dense_switch,
                           dense_density=dense_density)
    ws, nws = tw.workspace(T, D, F, C, K, dtype, train)
    y = torch.full((T, D), float("nan"), dtype=tdt, device="cuda")
    tw.twell_ffn_forward(dev["x"], dev["Wg"], dev["bg"], dev["rb"], dev["Wu"], dev["Wd"], D,
                         int(train), bufs.t, y, ws, nws)
    code, n_ovf = tw.twell_get_status(bufs.t)
    n_keep = min(n_ovf, bufs.cap)
    return dict(code=code, n_ovf=n_ovf, y=to_np64(y), ctl=ws[:24].cpu().numpy().copy(), idx=bufs.idx.cpu().numpy(),
                val=to_np64(bufs.val), nnz=bufs.nnz.cpu().numpy(),
                ovf_rows=bufs.ovf_rows[:n_keep].cpu().numpy(), g_fb=to_np64(bufs.g_fb[:n_keep]),
                u_val=None if bufs.u_val is None else to_np64(bufs.u_val),
                u_fb=None if bufs.u_fb is None else to_np64(bufs.u_fb[:n_keep]), bufs=bufs)


def check_forward(a, w, g, exact=False, rows=None, max_ambiguous=8):
    """Compare a GPU forward with the oracle on all rows (rows=None) or on the
    given sampled rows."""
    dt = w.dtype
    sel = np.arange(a["x"].shape[0]) if rows is None else np.asarray(rows)
    xs = a["x"][sel]
    rbs = None if a["rb"] is None else a["rb"][sel]
    z = oracle.gate(xs, a["Wg"], a["bg"], rbs, dt)
    ref = oracle.twell_pack(z, w.C, w.K, dt)
    if exact:
        band = np.full(z.shape, -1.0)
    else:
        band, _ = z_band(a, dt, rows=sel)
    gsub = dict(idx=g["idx"][:, sel, :], val=g["val"][:, sel, :], nnz=g["nnz"][:, sel])
    n_diff = compare_twell(gsub, ref, z, band, w.C, w.K, dt, max_ambiguous=max_ambiguous)
    if exact:
        assert n_diff == 0
        assert np.array_equal(gsub["val"], ref["val"])
    # overflow list: ascending, consistent with the GPU's own nnz, and equal to
    # the oracle's on the compared rows (up to ambiguous tiles)
    full_flags = row_ovf_from_nnz(g["nnz"], w.K)
    want_list = np.nonzero(full_flags)[0]
    assert g["n_ovf"] == len(want_list)
    assert np.array_equal(g["ovf_rows"], want_list[:len(g["ovf_rows"])])
    ref_flags = ref["row_ovf"].astype(bool)
    if exact:
        assert np.array_equal(full_flags[sel], ref_flags)
    # dense backup rows of overflow rows common to both
    pos = {int(t): i for i, t in enumerate(g["ovf_rows"])}
    for i_ref, t_sel in enumerate(np.nonzero(ref_flags)[0]):
        t = int(sel[t_sel])
        if t in pos:
            gr, rr = g["g_fb"][pos[t]], ref["g_fb"][i_ref]
            tol = (0 if exact else 2.0 ** -7) * np.abs(rr) + (0 if exact else 2 * band[t_sel])
            assert np.all(np.abs(gr - rr) <= tol), f"g_fb row {t}"
    y_ref = oracle.ffn_dense(xs, a["Wg"], a["bg"], rbs, a["Wu"], a["Wd"], dt, dt)
    assert np.isfinite(g["y"][sel]).all()
    extra = None if exact else value_allowance(a, dt, rows=sel, want=("y",))["y"]
    assert_close_rms(g["y"][sel], y_ref, dt, "y", extra=extra)
    return ref, z


# ------------------------------------------------------------ small cases --

def test_config1_full():
    w = synth.config1()
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    check_forward(a, w, g)


def test_bf16_gated_ragged_mixed_overflow():
    w = synth.Workload("mix", 300, 256, 1024, 128, 8, "bf16", True, -2.33, 7, hot_tokens=3,
                       seq_len=100, hot_bias=1.49)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    assert 3 <= g["n_ovf"] < 150      # the hot rows overflow, most rows do not
    check_forward(a, w, g)


def test_bf16_many_overflow_rows_gemm_path():
    """>= 128 overflow rows but fewer than half of all rows: the overflow rows
    run on the tensor-core dense-row GEMMs, the rest through TwELL."""
    w = synth.Workload("many", 600, 256, 1024, 128, 8, "bf16", True, -2.33, 16, hot_tokens=2,
                       seq_len=7, hot_bias=1.6)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0 and 128 <= g["n_ovf"] < 300
    check_forward(a, w, g)


def test_training_forward_stores_u():
    """train=1: u at the slots (u_val) and the u rows of overflow rows (u_fb),
    against x . W_up from the inputs, in hybrid and all-dense mode."""
    for bias, name in ((-2.33, "hyb"), (-1.0, "dense")):
        w = synth.Workload("tr" + name, 200, 256, 512, 64, 4, "bf16", True, bias, 17,
                           hot_tokens=2, seq_len=50, hot_bias=1.5)
        a = synth.generate(w)
        g = run_forward(a, w, train=True)
        assert g["code"] == 0
        u = synth.to_f64(a["x"], "bf16") @ synth.to_f64(a["Wu"], "bf16").T
        nt = w.F // w.C
        flags = row_ovf_from_nnz(g["nnz"], w.K)
        for j in range(nt):
            for t in np.nonzero(~flags)[0][:50]:
                k = min(int(g["nnz"][j, t]), w.K)
                cols = j * w.C + g["idx"][j, t, :k].astype(int)
                want = u[t, cols]
                assert np.all(np.abs(g["u_val"][j, t, :k] - want) <= 2.0 ** -7 * np.abs(want) + 1e-3)
        for i, t in enumerate(g["ovf_rows"][:20]):
            act = g["g_fb"][i] > 0
            want = u[t, act]
            assert np.all(np.abs(g["u_fb"][i][act] - want) <= 2.0 ** -7 * np.abs(want) + 1e-3)


def test_bf16_all_dense_mode():
    w = synth.Workload("dense", 200, 256, 512, 64, 4, "bf16", True, -1.0, 8)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0 and g["n_ovf"] > 100
    check_forward(a, w, g)


def test_integer_grid_bit_exact():
    T, D, F = 257, 320, 768
    rbu = np.zeros(T, dtype=np.int64)
    rbu[::50] = 120          # a few dense rows -> overflow
    a = synth.generate_grid(T, D, F, "bf16", True, 11, bias_units=-160, row_bias_units=rbu)
    w = synth.Workload("grid", T, D, F, 128, 8, "bf16", True, 0.0, 0)
    g = run_forward(a, w)
    assert g["code"] == 0 and g["n_ovf"] >= 1
    z = oracle.gate(a["x"], a["Wg"], a["bg"], a["rb"], "bf16")
    assert (z == 0).any(), "the grid case must contain exact ReLU ties"
    check_forward(a, w, g, exact=True)


@pytest.mark.parametrize("D", [512, 1024])
def test_bf16_dmodel_shapes(D):
    """d_model 512 (64 vectors per row: generic fused up/down path) and 1024
    (128 vectors: the exact-shape path, one vector per thread)."""
    w = synth.Workload(f"dm{D}", 200, D, 512, 128, 8, "bf16", True, -1.9, 30 + D // 512,
                       hot_tokens=2, seq_len=100, hot_bias=1.5)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0 and g["n_ovf"] >= 1
    check_forward(a, w, g)


@pytest.mark.parametrize("dt,D", [("bf16", 8192), ("f32", 4096)])
def test_maximum_dmodel(dt, D):
    """The largest d_model the ABI accepts (16 KB rows: 1024 vectors), with
    overflow rows (wide tiles) and a ragged token count; and the next size
    up is rejected."""
    w = synth.Workload(f"dmax{dt}", 70, D, 256, 64, 4, dt, True, -1.6, 48, hot_tokens=2,
                       seq_len=35, hot_bias=1.5)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0 and g["n_ovf"] >= 2
    check_forward(a, w, g)
    dtype = tw.TWELL_BF16 if dt == "bf16" else tw.TWELL_F32
    assert tw.twell_workspace_size(70, 2 * D, 256, 64, 4, dtype, 0) == 0


def test_fp32_dmodel1024_exact_shapes():
    """fp32 d_model 1024: 256 vectors per row, the exact-shape fused path."""
    w = synth.Workload("f32d1k", 96, 1024, 256, 64, 4, "f32", True, -1.7, 33)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    check_forward(a, w, g)


def _ctl(g):
    """(dense flag, slot counter) of the workspace's control block."""
    c = g["ctl"]
    return int(c[4:8].view(np.int32)[0]), int(c[16:24].view(np.uint64)[0])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_density_switch_runs_dense_rows(dtype):
    """~5% active with K = 16: few rows overflow, but the slots written exceed
    the default density threshold, so the whole forward runs on the dense
    path; with the test disabled the gathers run.  Both match the oracle; the
    slot counter equals sum(min(nnz, K)) exactly."""
    w = synth.Workload(f"dens{dtype}", 192, 256, 1024, 128, 16, dtype, True, -1.64, 34)
    a = synth.generate(w)
    on = run_forward(a, w, dense_density=0.0)
    off = run_forward(a, w, dense_density=-1.0)
    for g in (on, off):
        assert g["code"] == 0
        check_forward(a, w, g)
    dense_on, slots_on = _ctl(on)
    dense_off, slots_off = _ctl(off)
    expect = int(np.minimum(on["nnz"].astype(np.int64), w.K).sum())
    assert slots_on == expect and slots_off == expect
    assert expect > 0.013 * w.T * w.F
    assert dense_on == 1 and dense_off == 0


def test_density_switch_keeps_sparse_workloads_sparse():
    """1% active (the pages' regime): the default threshold keeps the gathers."""
    w = synth.Workload("dens1", 256, 256, 1024, 128, 8, "bf16", True, -2.33, 35)
    a = synth.generate(w)
    g = run_forward(a, w, dense_density=0.0)
    assert g["code"] == 0
    check_forward(a, w, g)
    dense, slots = _ctl(g)
    assert dense == 0 and 0 < slots < 0.013 * w.T * w.F


def test_fp32_gated_small_tiles():
    w = synth.Workload("f32g", 130, 64, 256, 32, 2, "f32", True, -1.6, 9)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    check_forward(a, w, g)


@pytest.mark.parametrize("C,K", [(32, 1), (32, 32), (64, 16), (128, 2)])
def test_bf16_tile_and_slot_shapes(C, K):
    w = synth.Workload(f"ck{C}_{K}", 96, 128, 512, C, K, "bf16", True, -1.9, 10 + K)
    a = synth.generate(w)
    g = run_forward(a, w, dense_switch=1.0)
    assert g["code"] == 0
    check_forward(a, w, g)


def test_capacity_error_keeps_y_correct():
    w = synth.Workload("cap", 128, 128, 512, 64, 2, "bf16", True, -1.3, 12)
    a = synth.generate(w)
    g = run_forward(a, w, ovf_cap=3, dense_switch=1.0)
    assert g["n_ovf"] > 3
    assert g["code"] == -4          # TWELL_ERR_CAPACITY
    assert len(g["ovf_rows"]) == 3
    dt = "bf16"
    y_ref = oracle.ffn_dense(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], dt, dt)
    assert_close_rms(g["y"], y_ref, dt, "y")


def test_single_token_and_empty_rows():
    w = synth.Workload("one", 1, 256, 512, 128, 8, "bf16", True, -2.33, 13)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    check_forward(a, w, g)
    w2 = synth.Workload("empty", 40, 256, 512, 128, 8, "bf16", True, -2.33, 14)
    a2 = synth.generate(w2)
    a2["rb"] = np.where(np.arange(40) % 2 == 0, -100.0, 0.0).astype(np.float32)
    g2 = run_forward(a2, w2)
    assert g2["code"] == 0
    assert (g2["nnz"][:, ::2] == 0).all() and (g2["y"][::2] == 0).all()
    check_forward(a2, w2, g2)


def test_nongated_bf16():
    w = synth.Workload("ng", 150, 256, 1024, 64, 4, "bf16", False, -2.0, 15)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    check_forward(a, w, g)


# --------------------------------------------------- full-size workloads --

def sample_rows(T, g, rng, n_rand=32, n_ovf=16):
    rows = set(range(16)) | set(range(T - 16, T))
    rows |= set(int(t) for t in g["ovf_rows"][:n_ovf])
    rows |= set(int(t) for t in rng.choice(T, size=n_rand, replace=False))
    return np.array(sorted(rows))


def test_config2_full_size_sampled():
    w = synth.config2()
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    assert g["n_ovf"] <= 20           # Binomial expectation ~1.6 rows
    rows = sample_rows(w.T, g, np.random.default_rng(2))
    check_forward(a, w, g, rows=rows)
    frac = float(np.minimum(g["nnz"], 255).sum()) / (w.T * w.F)
    assert abs(frac - 0.0099) < 0.001, frac


def test_config2_full_size_every_row():
    """Config 2 at full size, every token compared: the TwELL slots, counts
    and overflow list of all 4096 rows, and y over the whole tensor, so every
    tile of the persistent gate GEMM's grid and every token CTA of the
    gathers is checked, not a sample."""
    w = synth.config2()
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    # activity decisions whose exact z lies within fp32 rounding of 0 may go
    # either way: expected a few among the 33.5 M entries
    check_forward(a, w, g, max_ambiguous=64)


def test_config3_full_size_hot_rows():
    w = synth.config3()
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    hot = np.nonzero(a["rb"])[0]
    assert set(hot.tolist()) <= set(g["ovf_rows"].tolist())
    assert 256 <= g["n_ovf"] <= 300
    rows = sample_rows(w.T, g, np.random.default_rng(3), n_rand=24, n_ovf=8)
    check_forward(a, w, g, rows=rows)


@pytest.mark.parametrize("bias,K", [(-2.33, 8), (-1.28, 16), (-2.58, 4)])
def test_config4_points_sampled(bias, K):
    w = synth.config4(bias, K)
    a = synth.generate(w)
    g = run_forward(a, w)
    assert g["code"] == 0
    if bias == -1.28:
        assert g["n_ovf"] == w.T          # every row overflows: all-dense mode
    rows = sample_rows(w.T, g, np.random.default_rng(4), n_rand=12, n_ovf=4)[:48]
    check_forward(a, w, g, rows=rows)

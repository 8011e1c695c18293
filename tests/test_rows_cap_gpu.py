"""A workspace sized for a cap on the dense-path rows (twell_t.dense_rows_cap
with twell_workspace_size_rows): the dispatcher keeps the dense path within
the cap -- no all-dense mode when the cap is below T, overflow rows beyond it
stay on the gathers -- and the results still match the oracle; the backward
reports TWELL_ERR_CAPACITY when its overflow rows exceed the cap."""
import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import oracle
import synth
from twell_testlib import (assert_close_rms, check_backward, ctl_fields, to_np64, torch_dev,
                           value_allowance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    tw.load()


def run_capped(a, w, lam, cap, ovf_cap=None, dense_density=0.0):
    T, D, F, C, K = w.T, w.D, w.F, w.C, w.K
    d = {k: torch_dev(a[k]) for k in ("x", "Wg", "Wu", "Wd", "bg", "rb", "dy")}
    bufs = tw.TwellBuffers(T, F, C, K, tw.TWELL_BF16, ovf_cap, train=True,
                           dense_density=dense_density, dense_rows_cap=cap)
    ws, nws = tw.workspace(T, D, F, C, K, tw.TWELL_BF16, True, dense_rows_cap=cap)
    assert nws < tw.twell_workspace_size(T, D, F, C, K, tw.TWELL_BF16, 1)
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    tw.twell_ffn_forward(d["x"], d["Wg"], d["bg"], d["rb"], d["Wu"], d["Wd"], D, 1, bufs.t, y,
                         ws, nws)
    ctl_f = ws[:32].cpu().numpy().copy()
    code_f, n_ovf = tw.twell_get_status(bufs.t)
    dx = torch.empty_like(d["x"])
    dW = [torch.empty((F, D), dtype=torch.float32, device="cuda") for _ in range(3)]
    dbg = torch.empty((F,), dtype=torch.float32, device="cuda")
    tw.twell_ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], bufs.t, d["dy"], lam, D, dx, dW[0],
                          dbg, dW[1], dW[2], ws, nws)
    ctl_b = ws[:32].cpu().numpy().copy()
    code_b, _ = tw.twell_get_status(bufs.t)
    return dict(code_f=code_f, code_b=code_b, n_ovf=n_ovf, ctl_f=ctl_f, ctl_b=ctl_b,
                y=to_np64(y), dx=to_np64(dx), dWg=to_np64(dW[0]), dWu=to_np64(dW[1]),
                dWd=to_np64(dW[2]), dbg=to_np64(dbg))


def test_dense_regime_below_the_cap_stays_on_the_gathers():
    """~5% active (the density test would run every row densely) with a cap of
    128 rows: the forward and the backward keep every row on the gathers."""
    w = synth.Workload("cap5", 512, 256, 1024, 128, 16, "bf16", True, -1.64, 81, lam=1e-3,
                       train=True)
    a = synth.generate(w)
    g = run_capped(a, w, 1e-3, cap=128)
    assert g["code_f"] == 0 and g["code_b"] == 0
    assert ctl_fields(g["ctl_f"])[:2] == (0, 0) and ctl_fields(g["ctl_b"])[:2] == (0, 0)
    check_backward(a, w, g, 1e-3)


def test_overflow_rows_beyond_the_cap():
    """More overflow rows than the cap (>= 128, which would take the dense-row
    GEMMs): the forward runs them on the gathers from their wide tiles and y
    is complete; the backward, which keeps an overflow row's gradients in the
    workspace's dense-row buffers, reports a capacity error."""
    w = synth.Workload("capovf", 900, 256, 1024, 128, 8, "bf16", True, -2.33, 82, hot_tokens=2,
                       seq_len=7, hot_bias=1.6, lam=1e-3, train=True)
    a = synth.generate(w)
    g = run_capped(a, w, 1e-3, cap=256, dense_density=-1.0)
    n_rows, dense, n_ovf, ovf_gemm = ctl_fields(g["ctl_f"])
    assert n_ovf > 256 and (dense, ovf_gemm, n_rows) == (0, 0, 0)
    assert g["code_f"] == 0 and g["code_b"] == -4
    y_ref = oracle.ffn_dense(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], "bf16", "bf16")
    al = value_allowance(a, "bf16", want=("y",))
    assert_close_rms(g["y"], y_ref, "bf16", "y", extra=al["y"])


def test_overflow_rows_within_the_cap_take_the_dense_rows():
    """Overflow rows within the cap (and >= 128) take the dense-row GEMMs in
    the capped buffers, forward and backward."""
    w = synth.Workload("capin", 900, 256, 1024, 128, 8, "bf16", True, -2.33, 84, hot_tokens=2,
                       seq_len=7, hot_bias=1.6, lam=1e-3, train=True)
    a = synth.generate(w)
    g = run_capped(a, w, 1e-3, cap=384, dense_density=-1.0)
    assert g["code_f"] == 0 and g["code_b"] == 0
    for c in (g["ctl_f"], g["ctl_b"]):
        n_rows, dense, n_ovf, ovf_gemm = ctl_fields(c)
        assert 128 <= n_ovf <= 384 and (dense, ovf_gemm, n_rows) == (0, 1, n_ovf)
    check_backward(a, w, g, 1e-3)

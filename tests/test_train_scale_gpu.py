"""GPU parity of whole training steps at the pages' larger workload sizes,
through the C ABI, against the CPU oracle.

* d_model 4096 / d_ff 14336, T = 8192 (the sparsity sweep's shapes) in the
  dispatcher's regimes:
    - bias -2.58, K = 8 (~0.5% active, default thresholds): gathers forward
      and backward, dh from the gather SDDMM;
    - bias -2.33, K = 8 (~1% active, default thresholds): every row dense,
      forward and backward (the fp16 tensor-core path);
    - the same with the backward's density test off: the forward runs every
      row densely, the backward gathers with dh from the tensor-core GEMM
      read at the slots;
    - bias -1.64, K = 16 (~5% active): every row dense, forward and backward.
* T = 16384 with dense leading tokens (16 of every 1024 at ~20% active):
  the hot rows overflow into the dense backup on the forward and run on the
  dense-row path of the backward beside the gathers.

Samples are stratified so that every 128-row block of tokens and every TwELL
tile of neurons is compared (a fault confined to late row blocks, late tiles
or the second stream's work falls in the sample).  dbg is compared over every
neuron, which takes every token's gradient.  Entries whose fp32 activity the
GPU decided on the other side of 0 from the oracle (only allowed within the
order-error band) are left out with their row / neuron.
"""
import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import oracle
import synth
from twell_testlib import (activity_flips, assert_close_rms, check_backward, ctl_fields,
                           dh_gemm_of, run_train, value_allowance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    tw.load()


def stratified(n, block, seed, extra=()):
    """One random index in every block of `block` consecutive indices (and
    the given extra indices)."""
    rng = np.random.default_rng(seed)
    starts = np.arange(0, n, block)
    pick = starts + rng.integers(0, block, size=len(starts))
    return np.unique(np.concatenate([np.minimum(pick, n - 1), np.asarray(extra, dtype=np.int64)]))


def check_dbg_full(a, w, g, lam):
    """dbg over every neuron (every token's dz) against the oracle, leaving
    out neurons that hold an activity flip."""
    _, bad_n = activity_flips(a, w, g)
    cand = activity_flips.candidates
    assert len(bad_n) <= max(8, 2 * cand), (sorted(bad_n), cand)
    # (one token's dx comes along: the oracle takes explicit selections)
    b = oracle.ffn_backward(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], a["dy"], lam,
                            w.dtype, w.dtype, tok_sel=np.zeros(1, dtype=np.int32))
    keep = np.ones(w.F, dtype=bool)
    keep[sorted(bad_n)] = False
    al = value_allowance(a, w.dtype, lam=lam, rows=np.zeros(0, dtype=np.int64), want=("dbg",))
    assert_close_rms(g["dbg"][keep], b["dbg"][keep], w.dtype, "dbg(all neurons)", out_dtype="f32",
                     extra=al["dbg"][keep])


def check_y(a, w, g, rows):
    """The training forward's y on the given rows (activity flips change y
    only by an ambiguous gate value, below the bound)."""
    rb = None if a["rb"] is None else a["rb"][rows]
    y_ref = oracle.ffn_dense(a["x"][rows], a["Wg"], a["bg"], rb, a["Wu"], a["Wd"], w.dtype,
                             w.dtype)
    al = value_allowance(a, w.dtype, rows=rows, want=("y",))
    assert_close_rms(g["y"][rows], y_ref, w.dtype, "y", extra=al["y"])


REGIMES = {
    # name: (bias, K, backward density threshold (None: the forward's),
    #        forward all-dense, backward all-dense, dh GEMM, full dbg)
    "0.5pct_gathers": (-2.58, 8, None, 0, 0, 0, False),
    "1pct_all_dense": (-2.33, 8, 1e-9, 1, 1, 0, False),
    "1pct_dense_fwd_gather_bwd": (-2.33, 8, None, 1, 0, 1, True),
    "5pct_all_dense": (-1.64, 16, None, 1, 1, 0, False),
}


@pytest.mark.parametrize("regime", sorted(REGIMES))
def test_config4_training_step(regime):
    bias, K, bwd_dd, fwd_dense, bwd_dense, dh_gemm, full_dbg = REGIMES[regime]
    w = synth.scaled(synth.config4(bias, K), lam=1e-4, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, w.lam, dense_density=0.0, dh_density=0.0, out=out, keep_twell=True,
                  bwd_dense_density=bwd_dd)
    assert g["code"] == 0
    assert ctl_fields(out["ctl"])[1] == fwd_dense
    assert ctl_fields(out["ctl_bwd"])[1] == bwd_dense
    assert dh_gemm_of(out["ctl_bwd"]) == dh_gemm
    ts = stratified(w.T, 128, 400 + K, extra=(0, w.T - 1))
    ns = stratified(w.F, w.C, 500 + K, extra=(0, w.F - 1))
    check_y(a, w, g, ts)
    check_backward(a, w, g, w.lam, tok_sel=ts, neu_sel=ns, flips=True)
    if full_dbg:
        check_dbg_full(a, w, g, w.lam)
    for k in ("dx", "dWg", "dWu", "dWd", "dbg"):
        assert np.isfinite(g[k]).all(), k


def test_config3_training_step():
    """Dense leading tokens: the 256 hot rows (and a few others) overflow; the
    backward's dispatcher sends them to the dense-row GEMMs beside the
    gathers of every other row."""
    w = synth.scaled(synth.config3(), lam=1e-4, train=True)
    a = synth.generate(w)
    out = {}
    g = run_train(a, w, w.lam, dense_density=0.0, dh_density=0.0, out=out, keep_twell=True)
    assert g["code"] == 0
    n_rows, dense, n_ovf, ovf_gemm = ctl_fields(out["ctl_bwd"])
    assert dense == 0 and ovf_gemm == 1 and n_rows == n_ovf >= 256
    hot = np.nonzero(np.arange(w.T) % w.seq_len < w.hot_tokens)[0]
    assert set(hot.tolist()) <= set(g["ovf_rows"].tolist())
    rng = np.random.default_rng(33)
    ts = stratified(w.T, 128, 301, extra=rng.choice(hot, 12, replace=False))
    ns = stratified(w.F, w.C, 302)
    check_y(a, w, g, ts)
    check_backward(a, w, g, w.lam, tok_sel=ts, neu_sel=ns, flips=True)
    check_dbg_full(a, w, g, w.lam)


def test_config5_dbg_every_neuron():
    """The training-step workload (config 2 with dy, lambda = 1e-4): dbg of
    every neuron, i.e. the dz of every token, against the oracle."""
    w = synth.config5()
    a = synth.generate(w)
    g = run_train(a, w, w.lam, dense_density=0.0, dh_density=0.0, keep_twell=True)
    assert g["code"] == 0
    check_dbg_full(a, w, g, w.lam)
    ts = stratified(w.T, 128, 505)
    check_backward(a, w, g, w.lam, tok_sel=ts, neu_sel=stratified(w.F, w.C, 506), flips=True)

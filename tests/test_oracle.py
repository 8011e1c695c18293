"""Pins of the CPU oracle against what the pages and the mathematics fix.

The oracle is trusted only after these pass.  Each test checks the oracle
against something other than itself: a hand-worked case of the TwELL
definition, an independent numpy construction, a library routine (torch's
bf16 conversion, BLAS matmul), an identity the method relies on (sparse FFN ==
dense FFN), finite differences of the loss, or a closed form.
"""
import json
import os

import numpy as np
import pytest
import torch
from scipy.stats import norm

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- helpers --

def q_np(z, q):
    """Storage rounding done independently with torch casts (library routines)."""
    z = np.asarray(z, dtype=np.float64)
    if q == "none":
        return z.copy()
    z32 = torch.from_numpy(z).to(torch.float32)
    if q == "f32":
        return z32.double().numpy()
    return z32.to(torch.bfloat16).double().numpy()


def active_np(z, q):
    z = np.asarray(z, dtype=np.float64)
    if q == "none":
        return z > 0
    return z.astype(np.float32) > 0


def small_case(T, D, F, dt, gated, seed, bias, train=False, hot=None):
    w = synth.Workload("t", T, D, F, 4, 2, dt, gated, bias, seed, lam=0.0, train=train)
    a = synth.generate(w)
    if hot is not None:
        a["rb"] = np.asarray(hot, dtype=np.float32)
    return a


def f64(a, dt):
    return None if a is None else synth.to_f64(a, dt)


# ------------------------------------------------------------- rounding --

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-30),
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0, -0.0,
                  2.0 ** -126, 1e-40, 65504.0, 3.3895e38], dtype=np.float32),
    ])
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_round(v), want)
    assert np.array_equal(synth.f32_to_bf16_bits(v), want)
    # ties go to even: 1 + 2^-8 -> 1.0, 1 + 3*2^-8 -> 1 + 2^-6
    r = oracle.bf16_round(np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], dtype=np.float32))
    assert list(synth.bf16_bits_to_f32(r)) == [1.0, 1.0 + 2.0 ** -6]


# ------------------------------------------------------------------ gate --

@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_gate_matches_blas(dt):
    a = small_case(5, 7, 12, dt, True, 11, 0.1, hot=np.arange(5) * 0.25 - 0.5)
    z = oracle.gate(a["x"], a["Wg"], a["bg"], a["rb"], dt)
    x, W = f64(a["x"], dt), f64(a["Wg"], dt)
    want = x @ W.T + a["bg"].astype(np.float64)[None, :] + a["rb"].astype(np.float64)[:, None]
    np.testing.assert_allclose(z, want, rtol=1e-13, atol=1e-13)
    assert z.shape == (5, 12)


def test_gate_integer_grid_exact():
    a = synth.generate_grid(6, 64, 32, "bf16", True, 5, bias_units=-3,
                            row_bias_units=np.arange(6) - 2)
    z = oracle.gate(a["x"], a["Wg"], a["bg"], a["rb"], "bf16")
    xi = np.rint(f64(a["x"], "bf16")).astype(np.int64)
    Wi = np.rint(f64(a["Wg"], "bf16") * 16).astype(np.int64)
    want = (xi @ Wi.T - 3 + (np.arange(6) - 2)[:, None]) / 16.0
    assert np.array_equal(z, want)


# ------------------------------------------------------------------ pack --

def test_pack_hand_worked_case():
    g = json.load(open(os.path.join(HERE, "golden", "pack_tiny.json")))
    z = np.array(g["z"], dtype=np.float64)
    e = g["expect"]
    for q in ("none", "f32", "bf16"):
        tw = oracle.twell_pack(z, g["C"], g["K"], q)
        assert tw["nnz"].tolist() == e["nnz"]
        assert tw["idx"].tolist() == e["idx"]
        assert tw["val"].tolist() == e["val"]
        assert tw["row_ovf"].tolist() == e["row_ovf"]
        assert tw["ovf_rows"].tolist() == e["ovf_rows"]
        assert tw["g_fb"].tolist() == e["g_fb"]
        assert tw["n_ovf"] == 1


def test_pack_decision_and_value_rounding():
    z = np.array([[1e-50, 1e-40, -1e-50, 1.0 + 2.0 ** -8]], dtype=np.float64)
    tw = oracle.twell_pack(z, 4, 4, "bf16")
    # 1e-50 rounds to fp32 zero -> inactive; 1e-40 is an fp32 subnormal > 0.
    assert tw["nnz"].tolist() == [[2]]
    assert tw["idx"][0, 0].tolist() == [1, 3, 255, 255]
    assert tw["val"][0, 0, 1] == 1.0            # bf16 tie to even
    assert tw["val"][0, 0, 0] > 0
    tw32 = oracle.twell_pack(z, 4, 4, "f32")
    assert tw32["val"][0, 0, 1] == 1.0 + 2.0 ** -8
    twn = oracle.twell_pack(z, 4, 4, "none")
    assert twn["nnz"].tolist() == [[3]]
    assert twn["idx"][0, 0].tolist() == [0, 1, 3, 255]


@pytest.mark.parametrize("C,K,q,seed", [(4, 2, "none", 1), (8, 3, "bf16", 2), (16, 16, "f32", 3),
                                        (32, 1, "bf16", 4), (64, 8, "f32", 5), (128, 8, "bf16", 6)])
def test_pack_matches_independent_construction(C, K, q, seed):
    rng = np.random.default_rng(seed)
    T, F = 37, 256
    z = rng.standard_normal((T, F)) - 1.2
    z[rng.random((T, F)) < 0.05] = 0.0           # exact ReLU ties
    z[3, :] = 2.0                                  # a fully dense row
    z[5, :] = -1.0                                 # an empty row
    tw = oracle.twell_pack(z, C, K, q)
    nt = F // C
    act = active_np(z, q)
    zq = q_np(z, q)
    row_ovf = np.zeros(T, dtype=bool)
    for t in range(T):
        for j in range(nt):
            cols = np.nonzero(act[t, j * C:(j + 1) * C])[0]
            assert tw["nnz"][j, t] == len(cols)
            m = min(len(cols), K)
            assert tw["idx"][j, t, :m].tolist() == cols[:m].tolist()
            assert (tw["idx"][j, t, m:] == 255).all()
            assert tw["val"][j, t, :m].tolist() == zq[t, j * C + cols[:m]].tolist()
            assert (tw["val"][j, t, m:] == 0).all()
            assert (np.diff(tw["idx"][j, t, :m].astype(int)) > 0).all()
            assert (tw["val"][j, t, :m] > 0).all()
            row_ovf[t] |= len(cols) > K
    assert np.array_equal(tw["row_ovf"].astype(bool), row_ovf)
    assert tw["ovf_rows"].tolist() == np.nonzero(row_ovf)[0].tolist()
    relu_q = np.where(act, zq, 0.0)
    assert np.array_equal(tw["g_fb"], relu_q[row_ovf])
    # pack then unpack is the (rounded) ReLU output, bit for bit
    assert np.array_equal(oracle.twell_unpack(tw), relu_q)
    if K >= C:
        assert tw["n_ovf"] == 0


# ------------------------------------------------------------------- FFN --

def _ffn_numpy(a, dt, q):
    x, Wg, Wu, Wd = (f64(a[k], dt) for k in ("x", "Wg", "Wu", "Wd"))
    z = x @ Wg.T + a["bg"].astype(np.float64)[None, :]
    if a["rb"] is not None:
        z += a["rb"].astype(np.float64)[:, None]
    g = np.where(active_np(z, q), q_np(z, q), 0.0)
    h = g * (x @ Wu.T) if Wu is not None else g
    return h @ Wd, h


@pytest.mark.parametrize("dt,gated,q", [("f32", False, "f32"), ("bf16", True, "bf16"),
                                        ("f32", True, "none"), ("bf16", False, "bf16")])
def test_ffn_dense_matches_blas(dt, gated, q):
    a = small_case(9, 24, 40, dt, gated, 21, -0.3, hot=np.linspace(-0.5, 0.5, 9))
    y, h = oracle.ffn_dense(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], dt, q, want_h=True)
    y_np, h_np = _ffn_numpy(a, dt, q)
    np.testing.assert_allclose(h, h_np, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(y, y_np, rtol=1e-11, atol=1e-12 * np.abs(y_np).max())
    assert np.abs(y).max() > 0


@pytest.mark.parametrize("dt,gated,q,C,K", [("bf16", True, "bf16", 8, 2), ("f32", False, "f32", 16, 3),
                                            ("bf16", True, "bf16", 32, 8), ("f32", True, "none", 4, 1)])
def test_sparse_ffn_equals_dense_bit_exact(dt, gated, q, C, K):
    """The sparse FFN over TwELL + dense backup reproduces the dense FFN exactly:
    the dense loop only adds terms h = 0 in the same ascending order."""
    a = small_case(23, 32, 64, dt, gated, 31, -1.2, hot=np.where(np.arange(23) < 3, 1.5, 0.0))
    z = oracle.gate(a["x"], a["Wg"], a["bg"], a["rb"], dt)
    tw = oracle.twell_pack(z, C, K, q)
    assert tw["n_ovf"] > 0 and tw["n_ovf"] < 23
    y_sp = oracle.ffn_twell(a["x"], a["Wu"], a["Wd"], tw, dt)
    y_de = oracle.ffn_dense(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], dt, q)
    assert np.array_equal(y_sp, y_de)


# -------------------------------------------------------------- backward --

def _bwd_numpy(a, dt, q, lam):
    x, Wg, Wu, Wd, dy = (f64(a[k], dt) for k in ("x", "Wg", "Wu", "Wd", "dy"))
    z = x @ Wg.T + a["bg"].astype(np.float64)[None, :]
    if a["rb"] is not None:
        z += a["rb"].astype(np.float64)[:, None]
    act = active_np(z, q)
    g = np.where(act, q_np(z, q), 0.0)
    if Wu is not None:
        u = q_np(x @ Wu.T, q)  # u as saved for the backward, in the storage type
        h = g * u
    else:
        u = np.ones_like(g)
        h = g
    dh = dy @ Wd.T + lam * np.sign(h)
    dz = np.where(act, dh * u, 0.0)
    du = dh * g
    dx = dz @ Wg + (du @ Wu if Wu is not None else 0.0)
    return dict(dx=dx, dWg=dz.T @ x, dbg=dz.sum(0), dWu=(du.T @ x) if Wu is not None else None,
                dWd=h.T @ dy)


@pytest.mark.parametrize("dt,gated,q", [("bf16", True, "bf16"), ("f32", False, "f32"),
                                        ("f32", True, "none")])
def test_backward_matches_blas(dt, gated, q):
    a = small_case(11, 16, 48, dt, gated, 41, -0.4, train=True, hot=np.linspace(-1, 1, 11))
    lam = 0.01
    b = oracle.ffn_backward(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], a["dy"], lam, dt, q)
    want = _bwd_numpy(a, dt, q, lam)
    for k in ("dx", "dWg", "dbg", "dWu", "dWd"):
        if want[k] is None:
            assert b[k] is None
            continue
        scale = np.abs(want[k]).max()
        assert scale > 0
        np.testing.assert_allclose(b[k], want[k], rtol=1e-11, atol=1e-12 * scale, err_msg=k)


def test_backward_selection_is_row_subset():
    a = small_case(13, 16, 40, "bf16", True, 51, -0.5, train=True)
    full = oracle.ffn_backward(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], a["dy"], 1e-3,
                               "bf16", "bf16")
    ts, ns = np.array([12, 0, 5]), np.array([39, 2, 17, 3])
    sub = oracle.ffn_backward(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], a["dy"], 1e-3,
                              "bf16", "bf16", tok_sel=ts, neu_sel=ns)
    assert np.array_equal(sub["dx"], full["dx"][ts])
    for k in ("dWg", "dbg", "dWu", "dWd"):
        assert np.array_equal(sub[k], full[k][ns]), k


def _kink_free_case(gated, seed0):
    for seed in range(seed0, seed0 + 200):
        a = small_case(3, 5, 7, "f32", gated, seed, -0.2, train=True, hot=[0.1, -0.2, 0.3])
        x, Wg, Wu = (f64(a[k], "f32") for k in ("x", "Wg", "Wu"))
        z = x @ Wg.T + a["bg"].astype(np.float64)[None, :] + a["rb"].astype(np.float64)[:, None]
        h = np.where(z > 0, z, 0) * (x @ Wu.T if gated else 1.0)
        if np.abs(z).min() > 0.05 and np.abs(h[z > 0]).min() > 0.01 and (z > 0).sum() >= 4:
            return a
    raise RuntimeError("no kink-free case found")


@pytest.mark.parametrize("gated", [True, False])
def test_backward_finite_differences(gated):
    """Central differences of the loss (exact up to rounding for this piecewise
    quadratic function away from kinks) against the analytic gradient."""
    a = _kink_free_case(gated, 100 if gated else 300)
    lam = 0.05
    args = ["x", "Wg", "bg", "rb", "Wu", "Wd", "dy"]
    b = oracle.ffn_backward(*(a[k] for k in args), lam, "f32", "none")
    rng = np.random.default_rng(0)
    checks = [("x", "dx"), ("Wg", "dWg"), ("bg", "dbg"), ("Wd", "dWd")]
    if gated:
        checks.append(("Wu", "dWu"))
    for name, gname in checks:
        arr = a[name]
        for _ in range(4):
            i = tuple(rng.integers(0, s) for s in arr.shape)
            v = float(arr[i])
            hi, lo = np.float32(v + 1e-3), np.float32(v - 1e-3)
            Ls = []
            for pv in (hi, lo):
                b2 = dict(a)
                b2[name] = arr.copy()
                b2[name][i] = pv
                Ls.append(oracle.ffn_loss(*(b2[k] for k in args), lam, "f32", "none"))
            fd = (Ls[0] - Ls[1]) / (float(hi) - float(lo))
            an = b[gname][i]
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, i, fd, an)


def test_backward_closed_form_zero_down_weight():
    """With W_down = 0 the output gradient vanishes and dh = lambda*sign(h):
    dbg[n] = lambda * sum over active t of |u| (gated, sign(h) = sign(u))."""
    a = small_case(17, 8, 24, "f32", True, 61, -0.3, train=True)
    a["Wd"] = np.zeros_like(a["Wd"])
    lam = 0.25
    b = oracle.ffn_backward(a["x"], a["Wg"], a["bg"], None, a["Wu"], a["Wd"], a["dy"], lam, "f32", "f32")
    x, Wg, Wu = (f64(a[k], "f32") for k in ("x", "Wg", "Wu"))
    z = x @ Wg.T + a["bg"].astype(np.float64)
    u = (x @ Wu.T).astype(np.float32).astype(np.float64)  # u as saved (fp32 storage)
    want = lam * np.where(z.astype(np.float32) > 0, np.abs(u), 0.0).sum(0)
    np.testing.assert_allclose(b["dbg"], want, rtol=1e-12, atol=1e-14)
    assert np.abs(want).max() > 0
    np.testing.assert_array_equal(b["dWd"] != 0, (np.where(z.astype(np.float32) > 0, 1, 0).T @
                                                   np.abs(f64(a["dy"], "f32")) != 0))


# ------------------------------------------------------------- generator --

def test_generator_active_fraction_closed_form():
    """x ~ N(0,1), W ~ N(0,1/D) (variance) -> z ~ N(b, ~1): active = 1 - Phi(-b)."""
    w = synth.config2()
    a = synth.generate(synth.scaled(w, T=48, F=4096))
    x = torch.from_numpy(synth.bf16_bits_to_f32(a["x"]))
    W = torch.from_numpy(synth.bf16_bits_to_f32(a["Wg"]))
    z = (x @ W.T).numpy() + w.bias
    p = (z > 0).mean()
    want = 1 - norm.cdf(-w.bias)
    assert abs(want - 0.0099) < 1e-4
    assert abs(p - want) < 0.1 * want, (p, want)


def test_generator_hot_tokens():
    w = synth.scaled(synth.config3(), T=2048, F=1024)
    a = synth.generate(w)
    hot = np.nonzero(a["rb"])[0]
    assert hot.tolist() == list(range(16)) + list(range(1024, 1040))
    x = torch.from_numpy(synth.bf16_bits_to_f32(a["x"][hot]))
    W = torch.from_numpy(synth.bf16_bits_to_f32(a["Wg"]))
    z = (x @ W.T).numpy() + w.bias + a["rb"][hot, None]
    p = (z > 0).mean()
    assert abs(p - (1 - norm.cdf(0.84))) < 0.1 * 0.2, p


def test_generator_is_seeded_and_rows_prefix():
    w = synth.scaled(synth.config2(), T=16, D=256, F=512)
    a, b = synth.generate(w), synth.generate(w, rows=5)
    assert np.array_equal(a["x"][:5], b["x"]) and np.array_equal(a["Wd"], b["Wd"])

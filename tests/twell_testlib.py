"""Shared helpers of the parity tests: device upload, calls through the C ABI,
and comparisons against the oracle.

Tolerances (the stated precision of the method's outputs):
  y, dx, dW: max |a - ref| <= 2e-2 * rms(ref) (bf16) or 1e-4 * rms(ref) (fp32),
  with rms taken per output row (per token for y and dx, per neuron for dW),
  after allowing half an ulp of the output type at each element: rows differ
  in scale by ~5x between dense leading tokens and the rest, and the final
  bf16 rounding of the largest outputs alone (up to 2^-9 |y|) would break a
  bound that ignores the output type.
TwELL indices, counts and overflow lists: bit-exact, except where the fp32
sign of z is not fixed by the inputs: a (row, neuron) whose exact z lies
within the fp32 summation-error bound |z| <= band = D * 2^-23 * sum|x_d w_d|
+ 2^-22 (|bias| + |z|) may be decided either way (any fp32 summation order
stays inside that bound, twice the classical gamma_D bound).  Tiles and rows
that differ must contain such an ambiguous element, and they must be rare.
"""
from __future__ import annotations

import numpy as np

import synth

TOL = {"bf16": 2e-2, "f32": 1e-4}


def torch_dev(a, device="cuda"):
    import torch
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_np64(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def rms(a):
    return float(np.sqrt(np.mean(np.square(a)))) if a.size else 0.0


def half_ulp(ref, dtype):
    """Half a unit in the last place of the output type at each reference
    value: the error of the correctly rounded result, which every
    implementation storing its output in that type incurs."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    mant = 7 if dtype == "bf16" else 23
    e = np.floor(np.log2(np.maximum(ref, 1e-300)))
    return np.where(ref > 0, np.exp2(e - mant - 1), 0.0)


def assert_close_rms(got, ref, dtype, name, tol=None, out_dtype=None, extra=None):
    """max |got - ref| <= tol * rms(ref) per row of a 2-D output (a token's
    output vector, a neuron's weight-gradient row) and for 1-D outputs as a
    whole, after allowing half an ulp of the output type (out_dtype, default
    dtype) for the final store and, where given, a per-element allowance
    `extra` (the first-order effect of the fp32 uncertainty of z, see
    z_allowance).  Rows whose reference is exactly zero must be zero.
    Returns the worst ratio of the remaining error to rms."""
    tol = TOL[dtype] if tol is None else tol
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    od = dtype if out_dtype is None else out_dtype
    g2 = got.reshape(1, -1) if ref.ndim == 1 else got.reshape(ref.shape[0], -1)
    r2 = ref.reshape(1, -1) if ref.ndim == 1 else ref.reshape(ref.shape[0], -1)
    allow = half_ulp(r2, od)
    if extra is not None:
        allow = allow + np.asarray(extra, dtype=np.float64).reshape(r2.shape)
    excess = np.maximum(np.abs(g2 - r2) - allow, 0.0)
    err = np.max(excess, axis=1)
    r = np.sqrt(np.mean(np.square(r2), axis=1))
    bad = err > tol * r
    if bad.any():
        i = int(np.argmax(np.where(bad, err / np.maximum(r, 1e-300), 0)))
        raise AssertionError(f"{name}: row {i}: max|d|-allowance={err[i]:.3e} > {tol}*rms="
                             f"{tol * r[i]:.3e} ({int(bad.sum())} of {len(r)} rows)")
    return float(np.max(err / np.maximum(r, 1e-300)))


def z_band(a, dt, rows=None):
    """Per-element fp32 order-error bound of the gate pre-activation."""
    x = synth.to_f64(a["x"], dt)
    if rows is not None:
        x = x[rows]
    W = synth.to_f64(a["Wg"], dt)
    D = x.shape[1]
    s = np.abs(x) @ np.abs(W).T
    b = np.abs(a["bg"].astype(np.float64))[None, :]
    if a["rb"] is not None:
        rb = a["rb"].astype(np.float64)
        if rows is not None:
            rb = rb[rows]
        b = b + np.abs(rb)[:, None]
    return D * 2.0 ** -23 * s + 2.0 ** -22 * b, s


def z_allowance(a, dt, rows=None, lam=0.0):
    """First-order effect of the fp32 uncertainty of the gate pre-activation
    on the outputs.  Any fp32 implementation may compute z anywhere within
    +-band of the exact value (the same bound that governs the activity
    decisions); the gate value g = ReLU(z) inherits that uncertainty, and so
    does every output that is linear in g:
      y[t]   += sum_n band * |u| * |Wd[n]|          (plain FFN: u = 1)
      dWd[n] += sum_t band * |u| * |dy[t]|
      dWu[n] += sum_t band * |dh| * |x[t]|,  dx[t] += sum_n band * |dh| |Wu[n]|
    Returns a dict of these allowances for the rows `rows` (y, dx) and for all
    neurons (dW).  Negligible in bf16 (band ~ 1e-6 |z|), it matters in fp32
    where a small, cancellation-heavy z may differ by ~1e-4 relative."""
    f = lambda k: None if a[k] is None else synth.to_f64(a[k], dt)
    x, Wg, Wu, Wd = f("x"), f("Wg"), f("Wu"), f("Wd")
    sel = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    band, _ = z_band(a, dt)
    z = x @ Wg.T + a["bg"].astype(np.float64)[None, :]
    if a["rb"] is not None:
        z = z + a["rb"].astype(np.float64)[:, None]
    act = z.astype(np.float32) > 0
    u = x @ Wu.T if Wu is not None else np.ones_like(z)
    bu = band * np.abs(u) * act
    out = {"y": (bu @ np.abs(Wd))[sel]}
    if a.get("dy") is not None:
        dy = f("dy")
        dh = np.abs(dy @ Wd.T) + abs(lam)
        bd = band * dh * act
        out["dWd"] = bu.T @ np.abs(dy)
        out["dWu"] = bd.T @ np.abs(x)
        out["dx"] = ((bd @ np.abs(Wu)) if Wu is not None else np.zeros_like(x))[sel]
        out["dWg"] = np.zeros((Wg.shape[0], x.shape[1]))
        out["dbg"] = np.zeros(Wg.shape[0])
    return out


def decode_slots(idx, nnz, K):
    """Active local columns per (tile, row) from TwELL (complete only when nnz <= K)."""
    nt, T, _ = idx.shape
    out = {}
    for j in range(nt):
        for t in range(T):
            m = min(int(nnz[j, t]), K)
            out[(j, t)] = idx[j, t, :m].tolist()
    return out


def compare_twell(gpu, ref, z_ref, band, C, K, dt, rows=None, max_ambiguous=None):
    """Compare GPU TwELL (numpy arrays, possibly for a row subset) with the
    oracle's.  gpu/ref: dict with idx [nt][T][K], val, nnz [nt][T].
    Returns the number of (tile,row) pairs that differed (all ambiguous)."""
    nt, T, _ = ref["idx"].shape
    amb_el = np.abs(z_ref) <= band                      # [T][F]
    amb_tile = amb_el.reshape(T, nt, C).any(axis=2).T    # [nt][T]
    diff = (gpu["nnz"] != ref["nnz"]) | (gpu["idx"] != ref["idx"]).any(axis=2)
    bad = diff & ~amb_tile
    if bad.any():
        j, t = np.argwhere(bad)[0]
        raise AssertionError(
            f"TwELL mismatch at tile {j} row {t}: gpu nnz={gpu['nnz'][j, t]} idx={gpu['idx'][j, t]}"
            f" ref nnz={ref['nnz'][j, t]} idx={ref['idx'][j, t]}")
    same = ~diff
    # values at identical slots: within one bf16/fp32 rounding step of the
    # reference plus the order-error band
    gv, rv = gpu["val"][same], ref["val"][same]
    tol_rel = 2.0 ** -7 if dt == "bf16" else 2.0 ** -22
    bnd = np.repeat(np.maximum(band, 0).reshape(T, nt, C).max(axis=2).T[:, :, None], K, axis=2)[same]
    assert np.all(np.abs(gv - rv) <= tol_rel * np.abs(rv) + 2 * bnd + 1e-30), "TwELL values differ"
    n_diff = int(diff.sum())
    if max_ambiguous is not None:
        assert n_diff <= max_ambiguous, f"{n_diff} ambiguous tiles differ (> {max_ambiguous})"
    return n_diff


def row_ovf_from_nnz(nnz, K):
    return (nnz > K).any(axis=0)

"""Shared helpers of the parity tests: device upload, calls through the C ABI,
and comparisons against the oracle.

Tolerances (the stated precision of the method's outputs):
  y, dx, dW: max |a - ref| <= 2e-2 * rms(ref) (bf16) or 1e-4 * rms(ref) (fp32),
  asserted in two forms, each after allowing half an ulp of the output type
  at each element (the error of the correctly rounded result, which every
  implementation that stores its output in that type makes):
    - over the whole tensor compared (the bound as stated), and
    - per output row (per token for y and dx, per neuron for dW), which is
      stricter where rows differ in scale (dense leading tokens have ~5x
      larger outputs than the rest).
  Each output element also gets the first-order effect of the uncertainty
  of the activations g and u that both sides compute and store (see
  value_allowance): the fp32 rounding error of their sums (fp32 storage), or
  one bf16 ulp where a value lies within that error of a bf16 rounding
  midpoint (bf16 storage), and the worst-case band at entries whose activity
  is ambiguous (|z| within the band below).
TwELL indices, counts and overflow lists: bit-exact, except where the fp32
sign of z is not fixed by the inputs: a (row, neuron) whose exact z lies
within the fp32 summation-error bound |z| <= band = D * 2^-23 * sum|x_d w_d|
+ 2^-22 (|bias| + |z|) may be decided either way (any fp32 summation order
stays inside that bound, twice the classical gamma_D bound).  Tiles and rows
that differ must contain such an ambiguous element, and they must be rare.
"""
from __future__ import annotations

import json
import os

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


def _log_parity(name, dtype, tol, whole, worst_row, raw_whole):
    """Append the measured errors of one comparison to the file named by
    TWELL_PARITY_LOG (if set): the test, the output, and the ratios of the
    error (after the half-ulp allowance) to the bound's scale."""
    path = os.environ.get("TWELL_PARITY_LOG")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    with open(path, "a") as f:
        f.write(json.dumps({"test": test, "out": name, "dtype": dtype, "tol": tol,
                            "whole": whole, "worst_row": worst_row,
                            "whole_raw": raw_whole}) + "\n")


def assert_close_rms(got, ref, dtype, name, tol=None, out_dtype=None, extra=None):
    """The stated bound max |got - ref| <= tol * rms(ref), asserted over the
    whole compared tensor and per row of a 2-D output (a token's output
    vector, a neuron's weight-gradient row), after allowing half an ulp of
    the output type (out_dtype, default dtype) at each element and, where
    given, a per-element allowance `extra` (the first-order effect of the
    uncertainty of the stored activations, see value_allowance).  Rows whose
    reference is exactly zero must be zero.
    Returns the worst per-row ratio of the remaining error to rms."""
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
    diff = np.abs(g2 - r2)
    excess = np.maximum(diff - allow, 0.0)
    # whole tensor: the bound as stated
    rms_all = float(np.sqrt(np.mean(np.square(r2))))
    whole = float(excess.max()) / max(rms_all, 1e-300)
    raw_whole = float(diff.max()) / max(rms_all, 1e-300)
    if whole > tol:
        i, j = np.unravel_index(int(np.argmax(excess)), excess.shape)
        raise AssertionError(f"{name}: whole tensor: max|d|-allowance={excess[i, j]:.3e} at "
                             f"({i},{j}) > {tol}*rms={tol * rms_all:.3e}")
    # per row
    err = np.max(excess, axis=1)
    r = np.sqrt(np.mean(np.square(r2), axis=1))
    bad = err > tol * r
    if bad.any():
        i = int(np.argmax(np.where(bad, err / np.maximum(r, 1e-300), 0)))
        raise AssertionError(f"{name}: row {i}: max|d|-allowance={err[i]:.3e} > {tol}*rms="
                             f"{tol * r[i]:.3e} ({int(bad.sum())} of {len(r)} rows)")
    worst_row = float(np.max(err / np.maximum(r, 1e-300)))
    _log_parity(name, dtype if od == dtype else f"{dtype}->{od}", tol, whole, worst_row, raw_whole)
    return worst_row


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


def _stat_band(xs, W, D, bias_abs, v, s=None):
    """Six-sigma bound on the rounding error of an fp32 (or tensor-core,
    fp32-accumulated) sum v = xs . W[n] + bias: each of the D - 1 additions
    rounds by at most 2^-24 of a partial sum no larger than sum |x w| (s),
    the roundings independent and uniform."""
    if s is None:
        s = np.abs(xs) @ np.abs(W).T
    return 6.0 / np.sqrt(3.0) * np.sqrt(D) * 2.0 ** -24 * s + 2.0 ** -23 * (bias_abs + np.abs(v))


def _near_bf16_midpoint(v, e):
    """One bf16 ulp of v where v lies within e of a bf16 rounding midpoint
    (two implementations whose fp32 values differ by up to e may round it to
    neighbouring bf16 values), else 0."""
    a = np.abs(v)
    ex = np.floor(np.log2(np.maximum(a, 1e-300)))
    ulp = np.exp2(ex - 7)
    frac = a / ulp - np.floor(a / ulp)
    near = (np.abs(frac - 0.5) * ulp <= e) & (a > 0)
    return np.where(near, ulp, 0.0)


def value_allowance(a, dt, lam=0.0, rows=None, neurons=None, want=("y",), chunk=512):
    """First-order allowance for the uncertainty of the activations g (and,
    in the backward, u) that the GPU and the oracle each compute and store.
    An implementation sums z = x . W_gate[n] + b (and u = x . W_up[n]) in its
    own fp32 order (error e, a six-sigma bound, see _stat_band), so:
      - fp32 storage: g and u are known to within e;
      - bf16 storage: g and u are rounded to bf16; where the value lies
        within e of a rounding midpoint the two roundings are one ulp apart;
      - an activity-ambiguous entry (|z| within the worst-case band, where z
        may be taken on either side of 0) has g known to within the band.
    Propagated to the outputs (the backward consumes the stored g, u):
      y[t]    += sum_n dg |u| |Wd[n]|                  (plain FFN: u = 1)
      dx[t]   += sum_n |dh| du_ |Wg[n]| + |dh| dg |Wu[n]|
      dWg[n]  += sum_t |dh| du_ |x_t|,  dbg[n] += sum_t |dh| du_
      dWu[n]  += sum_t |dh| dg |x_t|,   dWd[n] += sum_t (|g| du_ + |u| dg) |dy_t|
    with dg, du_ the allowances of g and u (du_ = 0 for the plain FFN).
    rows / neurons select the token rows (y, dx) and neuron rows (dW, dbg)
    returned; None = all.  Token rows are processed in chunks."""
    f = lambda k: None if a[k] is None else synth.to_f64(a[k], dt)
    x, Wg, Wu, Wd = f("x"), f("Wg"), f("Wu"), f("Wd")
    dy = f("dy") if a.get("dy") is not None else None
    T, D = x.shape
    F = Wg.shape[0]
    bg = a["bg"].astype(np.float64)
    rb = None if a["rb"] is None else a["rb"].astype(np.float64)
    gated = Wu is not None
    tsel = np.arange(T) if rows is None else np.asarray(rows)
    nsel = np.arange(F) if neurons is None else np.asarray(neurons)
    out = {k: None for k in want}
    if "y" in want or "dx" in want:
        out_rows = {k: np.zeros((len(tsel), D)) for k in ("y", "dx") if k in want}
    acc_n = {k: np.zeros((len(nsel), D)) for k in ("dWg", "dWu", "dWd") if k in want}
    if "dbg" in want:
        acc_n["dbg"] = np.zeros(len(nsel))

    def entries(tok, ncols):
        """g, u, dh and the allowances dg, du_ of the (tok x ncols) block."""
        xs = x[tok]
        Wgn = Wg[ncols]
        b_abs = np.abs(bg[ncols])[None, :] + (0.0 if rb is None else np.abs(rb[tok])[:, None])
        z = xs @ Wgn.T + bg[ncols][None, :] + (0.0 if rb is None else rb[tok][:, None])
        act = z.astype(np.float32) > 0
        sg = np.abs(xs) @ np.abs(Wgn).T
        e_z = _stat_band(xs, Wgn, D, b_abs, z, sg)
        worst = D * 2.0 ** -23 * sg + 2.0 ** -22 * b_abs
        amb = np.abs(z) <= worst
        g = np.where(act, z, 0.0)
        if dt == "bf16":
            dg = _near_bf16_midpoint(g, e_z)
        else:
            dg = e_z.copy()
        dg = np.where(act, np.maximum(dg, np.where(amb, worst, 0.0)), 0.0)
        if gated:
            u = xs @ Wu[ncols].T
            e_u = _stat_band(xs, Wu[ncols], D, 0.0, u)
            du_ = (_near_bf16_midpoint(u, e_u) if dt == "bf16" else e_u) * act
        else:
            u = np.ones_like(z)
            du_ = np.zeros_like(z)
        dh = None
        if dy is not None:
            dh = np.abs(dy[tok] @ Wd[ncols].T) + abs(lam)
        return g, u, dg, du_, dh

    if "y" in want or "dx" in want:
        for c0 in range(0, len(tsel), chunk):
            tok = tsel[c0:c0 + chunk]
            g, u, dg, du_, dh = entries(tok, np.arange(F))
            if "y" in want:
                out_rows["y"][c0:c0 + chunk] = (dg * np.abs(u)) @ np.abs(Wd)
            if "dx" in want:
                m = dh * du_ @ np.abs(Wg)
                if gated:
                    m = m + (dh * dg) @ np.abs(Wu)
                out_rows["dx"][c0:c0 + chunk] = m
        for k in out_rows:
            out[k] = out_rows[k]
    if acc_n:
        for c0 in range(0, T, chunk):
            tok = np.arange(c0, min(T, c0 + chunk))
            g, u, dg, du_, dh = entries(tok, nsel)
            ax = np.abs(x[tok])
            if "dWg" in acc_n:
                acc_n["dWg"] += (dh * du_).T @ ax
            if "dbg" in acc_n:
                acc_n["dbg"] += (dh * du_).sum(axis=0)
            if "dWu" in acc_n and gated:
                acc_n["dWu"] += (dh * dg).T @ ax
            if "dWd" in acc_n:
                acc_n["dWd"] += (np.abs(g) * du_ + np.abs(u) * dg).T @ np.abs(dy[tok])
        out.update(acc_n)
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


# ------------------------------------------------- training-step helpers --

def shifted(t, elems):
    """A copy of device tensor t whose data starts `elems` elements past an
    allocation boundary (16-byte aligned but not 32-byte aligned for 8 bf16)."""
    import torch
    buf = torch.empty(t.numel() + elems, dtype=t.dtype, device=t.device)
    v = buf[elems:].view(t.shape)
    v.copy_(t)
    return v


def run_train(a, w, lam, ovf_cap=None, dense_density=-1.0, out=None, wd_shift=0, dh_density=-1.0,
              keep_twell=False, bwd_dense_density=None, gather_passes=0):
    """Forward (train) + backward through the C ABI.  dense_density < 0 keeps
    the density test of the dispatcher off, so that moderately dense test
    workloads still run the gather kernels; dh_density < 0 keeps dh on the
    gather SDDMM (> 0: on the tensor-core GEMM read at the slots above that
    density; 0: the dispatcher's default); out (dict) receives the
    workspace's control block after the forward ("ctl") and after the
    backward ("ctl_bwd").  keep_twell: also return the saved TwELL (idx, nnz,
    the overflow rows and their dense backup rows) for activity checks.
    bwd_dense_density: the backward's own density threshold (the twell_t is
    passed per call), else the forward's.  gather_passes: the twell_t's
    passes of the gather kernels (0: the library's choice)."""
    import torch
    import activation_sparse_transformer_gate_gb300 as tw
    T, D, F, C, K = a["x"].shape[0], a["x"].shape[1], a["Wg"].shape[0], w.C, w.K
    dtype = tw.TWELL_BF16 if w.dtype == "bf16" else tw.TWELL_F32
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    d = {k: torch_dev(a[k]) for k in ("x", "Wg", "Wu", "Wd", "bg", "rb", "dy")}
    if wd_shift:
        d["Wd"] = shifted(d["Wd"], wd_shift)
    bufs = tw.TwellBuffers(T, F, C, K, dtype, ovf_cap, train=True, dense_density=dense_density,
                           dh_density=dh_density, gather_passes=gather_passes)
    ws, nws = tw.workspace(T, D, F, C, K, dtype, True)
    y = torch.empty((T, D), dtype=tdt, device="cuda")
    tw.twell_ffn_forward(d["x"], d["Wg"], d["bg"], d["rb"], d["Wu"], d["Wd"], D, 1, bufs.t, y, ws, nws)
    if out is not None:
        out["ctl"] = ws[:32].cpu().numpy().copy()
    dx = torch.full((T, D), float("nan"), dtype=tdt, device="cuda")
    dWg = torch.full((F, D), float("nan"), dtype=torch.float32, device="cuda")
    dWu = torch.full_like(dWg, float("nan")) if d["Wu"] is not None else None
    dWd = torch.full_like(dWg, float("nan"))
    dbg = torch.full((F,), float("nan"), dtype=torch.float32, device="cuda")
    if bwd_dense_density is not None:
        bufs.t.dense_density = float(bwd_dense_density)
    tw.twell_ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], bufs.t, d["dy"], lam, D, dx, dWg, dbg,
                          dWu, dWd, ws, nws)
    if out is not None:
        out["ctl_bwd"] = ws[:32].cpu().numpy().copy()
    code, n_ovf = tw.twell_get_status(bufs.t)
    r = dict(code=code, n_ovf=n_ovf, y=to_np64(y), dx=to_np64(dx), dWg=to_np64(dWg),
             dbg=to_np64(dbg), dWu=None if dWu is None else to_np64(dWu), dWd=to_np64(dWd))
    if keep_twell:
        n_keep = min(n_ovf, bufs.cap)
        r.update(idx=bufs.idx.cpu().numpy(), nnz=bufs.nnz.cpu().numpy(),
                 ovf_rows=bufs.ovf_rows[:n_keep].cpu().numpy(),
                 g_fb=to_np64(bufs.g_fb[:n_keep]), C=C, K=K)
    return r


def ctl_fields(c):
    """(n_rows, dense, n_ovf, ovf_gemm) of a saved control block."""
    return tuple(int(v) for v in c[:16].view(np.int32))


def dh_gemm_of(c):
    """The backward's choice of the tensor-core dh GEMM in a saved control block."""
    return int(c[24:28].view(np.int32)[0])


def gpu_activity(g, rows):
    """[len(rows)][F] activity of the given rows as the GPU's saved TwELL holds
    it: the slots of a row whose tiles all fit K, the dense backup row of an
    overflow row."""
    idx, nnz, C, K = g["idx"], g["nnz"], g["C"], g["K"]
    nt, T, _ = idx.shape
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), nt * C), dtype=bool)
    sub = idx[:, rows, :].astype(np.int64)                      # [nt][R][K]
    live = np.arange(K)[None, None, :] < np.minimum(nnz[:, rows], K)[:, :, None]
    j, r, _ = np.nonzero(live)
    out[r, j * C + sub[live]] = True
    pos = {int(t): i for i, t in enumerate(g["ovf_rows"])}
    for q, t in enumerate(rows):
        if int(t) in pos:
            out[q] = g["g_fb"][pos[int(t)]] > 0
    return out


def gpu_activity_cols(g, neurons):
    """[T][len(neurons)] activity of the given neurons in every row, as the
    GPU's saved TwELL holds it."""
    idx, nnz, C, K = g["idx"], g["nnz"], g["C"], g["K"]
    nt, T, _ = idx.shape
    ovf = set(int(t) for t in g["ovf_rows"])
    out = np.zeros((T, len(neurons)), dtype=bool)
    for q, n in enumerate(neurons):
        j, c = int(n) // C, int(n) % C
        m = np.minimum(nnz[j], K)
        hit = (idx[j] == c) & (np.arange(K)[None, :] < m[:, None])
        out[:, q] = hit.any(axis=1)
    for i, t in enumerate(g["ovf_rows"]):
        out[int(t)] = g["g_fb"][i][np.asarray(neurons, dtype=np.int64)] > 0
    return out


def activity_flips(a, w, g, rows=None, neurons=None, chunk=1024):
    """Entries whose activity the GPU decided differently from the oracle
    (z > 0 in fp32).  Such an entry must be activity-ambiguous: its exact z
    lies within the fp32 order-error band.  Returns the set of rows (of
    `rows`) and of neurons (of `neurons`) that hold a flipped entry;
    rows=None / neurons=None check every row / every neuron (in chunks of
    tokens)."""
    dt = w.dtype
    T = a["x"].shape[0]
    bad_rows, bad_neurons = set(), set()
    cand = [0]

    def check(zz, act_gpu, tok, neu):
        act_ref = zz.astype(np.float32) > 0
        # entries within (twice) the statistical fp32 band of 0, estimated on
        # a few rows of the block: the only ones whose activity any
        # implementation may realistically take the other way
        xs = synth.to_f64(a["x"][tok[:4]], dt)
        W = synth.to_f64(a["Wg"][neu], dt)
        tau = 2.0 * float(np.median(_stat_band(xs, W, xs.shape[1], 0.0, 0.0)))
        cand[0] += int((np.abs(zz) <= tau).sum())
        diff = np.argwhere(act_ref != act_gpu)
        for r, c in diff:
            t, n = int(tok[r]), int(neu[c])
            x = synth.to_f64(a["x"][t], dt)
            W = synth.to_f64(a["Wg"][n], dt)
            rb = 0.0 if a["rb"] is None else abs(float(a["rb"][t]))
            band = len(x) * 2.0 ** -23 * float(np.abs(x) @ np.abs(W)) + \
                2.0 ** -22 * (abs(float(a["bg"][n])) + rb)
            assert abs(zz[r, c]) <= band, f"activity of ({t},{n}) differs at z={zz[r, c]:.3e}"
            bad_rows.add(t)
            bad_neurons.add(n)

    import oracle
    if rows is not None:
        rows = np.asarray(rows)
        rb = None if a["rb"] is None else a["rb"][rows]
        zz = oracle.gate(a["x"][rows], a["Wg"], a["bg"], rb, dt)
        check(zz, gpu_activity(g, rows), rows, np.arange(a["Wg"].shape[0]))
    if neurons is not None:
        neurons = np.asarray(neurons)
        zz = oracle.gate(a["x"], a["Wg"][neurons], a["bg"][neurons], a["rb"], dt)
        check(zz, gpu_activity_cols(g, neurons), np.arange(T), neurons)
    if rows is None and neurons is None:
        F = a["Wg"].shape[0]
        for t0 in range(0, T, chunk):
            tok = np.arange(t0, min(T, t0 + chunk))
            rb = None if a["rb"] is None else a["rb"][tok]
            zz = oracle.gate(a["x"][tok], a["Wg"], a["bg"], rb, dt)
            check(zz, gpu_activity(g, tok), tok, np.arange(F))
    activity_flips.candidates = cand[0]
    return bad_rows, bad_neurons


def check_backward(a, w, g, lam, tok_sel=None, neu_sel=None, flips=False, max_flips=3):
    """dx on tok_sel (all rows when None) and dWg, dWu, dWd, dbg on neu_sel
    (all neurons when None) against the oracle.  flips=True (needs the saved
    TwELL in g): rows and neurons holding an entry whose activity the GPU
    took on the other side of 0 from the oracle (an ambiguous fp32 decision,
    checked to lie within the order-error band; dz = [z > 0] dh u jumps
    there) are left out of the comparison, at most max_flips of each."""
    import oracle
    dt = w.dtype
    b = oracle.ffn_backward(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], a["dy"], lam, dt,
                            dt, tok_sel=tok_sel, neu_sel=neu_sel)
    T, F = a["x"].shape[0], a["Wg"].shape[0]
    ts = np.arange(T) if tok_sel is None else np.asarray(tok_sel)
    ns = np.arange(F) if neu_sel is None else np.asarray(neu_sel)
    keep_t = np.ones(len(ts), dtype=bool)
    keep_n = np.ones(len(ns), dtype=bool)
    if flips:
        br, _ = activity_flips(a, w, g, rows=ts)
        cr = activity_flips.candidates
        _, bn = activity_flips(a, w, g, neurons=ns)
        cn = activity_flips.candidates
        assert len(br) <= max(max_flips, 2 * cr), (sorted(br), cr)
        assert len(bn) <= max(max_flips, 2 * cn), (sorted(bn), cn)
        keep_t = ~np.isin(ts, sorted(br))
        keep_n = ~np.isin(ns, sorted(bn))
    want = ("dx", "dWg", "dWd", "dbg") + (("dWu",) if a["Wu"] is not None else ())
    al = value_allowance(a, dt, lam=lam, rows=ts, neurons=ns, want=want)
    ex = al.get("dx")
    assert_close_rms(g["dx"][ts][keep_t], b["dx"][keep_t], dt, "dx",
                     extra=None if ex is None else ex[keep_t])
    for k in ("dWg", "dWd", "dbg") + (("dWu",) if a["Wu"] is not None else ()):
        ex = al.get(k)
        assert_close_rms(g[k][ns][keep_n], b[k][keep_n], dt, k, out_dtype="f32",
                         extra=None if ex is None else ex[keep_n])
    # neurons that are never active have exactly zero gradient rows
    dead = np.all(b["dWd"] == 0, axis=1) & keep_n
    if dead.any():
        assert np.all(g["dWg"][ns][dead] == 0) and np.all(g["dWd"][ns][dead] == 0)
        assert np.all(g["dbg"][ns][dead] == 0)
    return b

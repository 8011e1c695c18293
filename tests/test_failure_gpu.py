"""Failure detection on the GPU without a fault.

* Bounded waits: the tensor-core kernels give up a pipeline wait after a
  limit, record TWELL_ERR_TIMEOUT, wait for their own copies and MMAs in
  flight, free their TMEM and return.  The test-only build
  ``libtwell_timeout.so`` sets that limit to 1 ns, so on a sane input the
  first wait that is not satisfied at once runs out.  It runs in a child
  process: each entry point must return, report the timeout through the
  status word, and leave the CUDA context usable (a later call of the same
  library still computes a correct result).
* Malformed TwELL: a live slot whose index is >= C, handed to the backward,
  is reported as TWELL_ERR_INDEX by every path that reads slots (gather dh,
  tensor-core dh read at the slots, dense-path rows), and the call returns.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import synth
from twell_testlib import torch_dev

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TIMEOUT_CHILD = textwrap.dedent(r"""
    import ctypes, sys
    import numpy as np
    import torch
    sys.path.insert(0, sys.argv[1])
    import activation_sparse_transformer_gate_gb300 as tw
    from activation_sparse_transformer_gate_gb300 import _build
    import synth

    lib = tw.load(_build.lib_path("timeout"))
    torch.cuda.set_device(0)
    sh = torch.cuda.current_stream().cuda_stream
    w = synth.Workload("to", 256, 512, 1024, 128, 8, "bf16", True, -2.33, 91, hot_tokens=2,
                       seq_len=64, hot_bias=1.5, train=True)
    a = synth.generate(w)

    def dev(v):
        if v is None:
            return None
        if v.dtype == np.uint16:
            return torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(v).cuda()

    d = {k: dev(a[k]) for k in ("x", "Wg", "Wu", "Wd", "bg", "rb", "dy")}
    P = lambda t: None if t is None else t.data_ptr()

    def buffers(**kw):
        b = tw.TwellBuffers(w.T, w.F, w.C, w.K, tw.TWELL_BF16, train=True, **kw)
        for t in (b.idx, b.val, b.nnz, b.ovf_rows, b.g_fb, b.u_val, b.u_fb):
            t.zero_()
        return b

    def status(b):
        n = ctypes.c_int32(0)
        return lib.twell_get_status(ctypes.byref(b.t), sh, ctypes.byref(n))

    nws = lib.twell_workspace_size(w.T, w.D, w.F, w.C, w.K, tw.TWELL_BF16, 1)
    ws = torch.zeros((nws,), dtype=torch.uint8, device="cuda")
    y = torch.zeros((w.T, w.D), dtype=torch.bfloat16, device="cuda")
    dx = torch.zeros_like(y)
    dW = [torch.zeros((w.F, w.D), dtype=torch.float32, device="cuda") for _ in range(3)]
    dbg = torch.zeros((w.F,), dtype=torch.float32, device="cuda")
    out = []

    # 1. the gate GEMM with the TwELL epilogue alone
    b = buffers()
    rc = lib.twell_pack(P(d["x"]), P(d["Wg"]), P(d["bg"]), P(d["rb"]), w.D, ctypes.byref(b.t),
                        P(ws), nws, sh)
    out.append(("pack", rc, status(b), status(b)))
    # 2. training step with every row on the dense path (all GEMM epilogues) and
    # 3. with the gathers and dh from the GEMM read at the slots
    for name, kw in (("all_dense", dict(dense_density=1e-9)),
                     ("dh_gemm", dict(dense_density=-1.0, dh_density=1e-9))):
        b = buffers(**kw)
        rc1 = lib.twell_ffn_forward(P(d["x"]), P(d["Wg"]), P(d["bg"]), P(d["rb"]), P(d["Wu"]),
                                    P(d["Wd"]), w.D, 1, ctypes.byref(b.t), P(y), P(ws), nws, sh)
        rc2 = lib.twell_ffn_backward(P(d["x"]), P(d["Wg"]), P(d["Wu"]), P(d["Wd"]),
                                     ctypes.byref(b.t), P(d["dy"]), ctypes.c_float(1e-4), w.D,
                                     P(dx), P(dW[0]), P(dbg), P(dW[1]), P(dW[2]), P(ws), nws, sh)
        out.append((name, rc1 * 100 + rc2, status(b), status(b)))
    torch.cuda.synchronize()

    # the context is still usable: the same library packs a dense matrix
    # (no pipeline waits on that path) and the result is exact
    H = np.where(np.random.default_rng(5).random((w.T, w.F)) < 0.02, 1.0, 0.0).astype(np.float32)
    Ht = torch.from_numpy(H).to(torch.bfloat16).cuda()
    b = buffers()
    rc = lib.twell_pack_dense(P(Ht), ctypes.byref(b.t), sh)
    st = status(b)
    nnz = b.nnz.cpu().numpy().astype(np.int64)
    want = (H.reshape(w.T, w.F // w.C, w.C) > 0).sum(axis=2).T
    out.append(("after", rc, st, int(np.array_equal(nnz, want))))
    for r in out:
        print("RESULT", *r)
""")


def test_bounded_waits_time_out_and_leave_the_context_usable():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build(variants=("timeout",))
    r = subprocess.run([sys.executable, "-c", TIMEOUT_CHILD, ROOT], capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = {ln.split()[1]: [int(v) for v in ln.split()[2:]] for ln in r.stdout.splitlines()
           if ln.startswith("RESULT")}
    for name in ("pack", "all_dense", "dh_gemm"):
        rc, first, second = res[name]
        assert rc == 0, (name, rc)                   # launches succeeded, calls returned
        assert first == -6, (name, first)            # TWELL_ERR_TIMEOUT in the status word
        assert second == 0, (name, second)           # read once, then cleared
    rc, st, exact = res["after"]
    assert rc == 0 and st == 0 and exact == 1


# ---------------------------------------------------------------- index --

@pytest.fixture(scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    tw.load()


def _train_case(w, lam, **kw):
    a = synth.generate(w)
    dtype = tw.TWELL_BF16 if w.dtype == "bf16" else tw.TWELL_F32
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    d = {k: torch_dev(a[k]) for k in ("x", "Wg", "Wu", "Wd", "bg", "rb", "dy")}
    bufs = tw.TwellBuffers(w.T, w.F, w.C, w.K, dtype, train=True, **kw)
    ws, nws = tw.workspace(w.T, w.D, w.F, w.C, w.K, dtype, True)
    y = torch.empty((w.T, w.D), dtype=tdt, device="cuda")
    tw.twell_ffn_forward(d["x"], d["Wg"], d["bg"], d["rb"], d["Wu"], d["Wd"], w.D, 1, bufs.t, y,
                         ws, nws)
    code, _ = tw.twell_get_status(bufs.t)
    assert code == 0
    dx = torch.empty_like(d["x"])
    dW = [torch.empty((w.F, w.D), dtype=torch.float32, device="cuda") for _ in range(3)]
    dbg = torch.empty((w.F,), dtype=torch.float32, device="cuda")

    def backward():
        tw.twell_ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], bufs.t, d["dy"], lam, w.D, dx,
                              dW[0], dbg, dW[1] if d["Wu"] is not None else None, dW[2], ws, nws)
        return tw.twell_get_status(bufs.t)[0]

    return bufs, backward, dx, dW, dbg


def _corrupt_live_slot(bufs, C, K):
    """Set the index of one live slot of a non-overflow row to C + 3 (a value
    no tile holds); returns (tile, row, slot, old index)."""
    nnz = bufs.nnz.cpu().numpy()
    ovf = (nnz > K).any(axis=0)
    for j in range(nnz.shape[0]):
        for t in np.nonzero(~ovf & (nnz[j] > 0))[0]:
            old = int(bufs.idx[j, t, 0].item())
            bufs.idx[j, t, 0] = C + 3
            return j, int(t), 0, old
    raise AssertionError("no live slot")


@pytest.mark.parametrize("path", ["sddmm", "dh_gemm", "dense_rows", "f32"])
def test_malformed_index_is_reported(_lib, path):
    if path == "f32":
        w = synth.scaled(synth.config1(), train=True, T=128)
        kw = dict(dense_density=-1.0, dh_density=-1.0)
        lam = 1e-3
    else:
        w = synth.Workload("ix", 256, 256, 1024, 128, 8, "bf16", True, -2.0, 97, train=True)
        kw = {"sddmm": dict(dense_density=-1.0, dh_density=-1.0),
              "dh_gemm": dict(dense_density=-1.0, dh_density=1e-9),
              "dense_rows": dict(dense_density=1e-9)}[path]
        lam = 1e-4
    bufs, backward, dx, dW, dbg = _train_case(w, lam, **kw)
    clean = backward()
    assert clean == 0
    ref = [t.clone() for t in (dx, dW[0], dW[2], dbg)]
    j, t, k, old = _corrupt_live_slot(bufs, w.C, w.K)
    assert backward() == -5                            # TWELL_ERR_INDEX
    bufs.idx[j, t, k] = old                            # repaired: same results as before
    assert backward() == 0
    for a, b in zip(ref, (dx, dW[0], dW[2], dbg)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("scale, want", [(16.0, -11), (1.0, 0)])
def test_fp16_range_is_reported(_lib, scale, want):
    """The dense-path GEMMs take fp16 operands: h = g u beyond 65504 (x = 16,
    unit weights, d_model 64: g = u = 1024) is refused with TWELL_ERR_RANGE;
    the same call with x = 1 (h = 4096) runs clean."""
    T, D, F, C, K = 128, 64, 256, 64, 8
    bf = torch.bfloat16
    x = torch.full((T, D), scale, dtype=bf, device="cuda")
    Wg = torch.ones((F, D), dtype=bf, device="cuda")
    Wu = torch.ones((F, D), dtype=bf, device="cuda")
    Wd = torch.full((F, D), 1.0 / 256, dtype=bf, device="cuda")
    bg = torch.zeros((F,), dtype=torch.float32, device="cuda")
    bufs = tw.TwellBuffers(T, F, C, K, tw.TWELL_BF16, dense_density=1e-9)
    ws, nws = tw.workspace(T, D, F, C, K, tw.TWELL_BF16, False)
    y = torch.empty((T, D), dtype=bf, device="cuda")
    tw.twell_ffn_forward(x, Wg, bg, None, Wu, Wd, D, 0, bufs.t, y, ws, nws)
    code, n_ovf = tw.twell_get_status(bufs.t)
    assert n_ovf == T            # every tile holds 64 > K active columns
    assert code == want
    if want == 0:                # h = 4096 at every entry: y = 4096 * 256 / 256
        assert torch.equal(y, torch.full_like(y, 4096.0))

"""GPU parity of the two packing entry points: twell_pack_dense (bit-exact on
any input: no arithmetic decides anything) and twell_pack (gate GEMM + ReLU +
TwELL epilogue + hybrid split + dense backup rows)."""
import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import oracle
import synth
from twell_testlib import compare_twell, to_np64, torch_dev, z_band

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    tw.load()


def read(bufs, n):
    k = min(n, bufs.cap)
    return dict(idx=bufs.idx.cpu().numpy(), val=to_np64(bufs.val), nnz=bufs.nnz.cpu().numpy(),
                ovf_rows=bufs.ovf_rows[:k].cpu().numpy(), g_fb=to_np64(bufs.g_fb[:k]))


@pytest.mark.parametrize("dt,C,K,T,F,p_act", [("bf16", 128, 8, 333, 1024, 0.05),
                                              ("f32", 64, 4, 97, 512, 0.08),
                                              ("bf16", 32, 1, 64, 256, 0.03),
                                              ("bf16", 128, 32, 50, 512, 0.3)])
def test_pack_dense_bit_exact(dt, C, K, T, F, p_act):
    rng = np.random.default_rng(T + F + K)
    H = rng.standard_normal((T, F)).astype(np.float32)
    H = np.where(rng.random((T, F)) < p_act, np.abs(H), 0.0).astype(np.float32)
    H[7 % T, :] = 1.0                                  # a full row
    if dt == "bf16":
        Hs = synth.f32_to_bf16_bits(H)
        Hd = synth.bf16_bits_to_f32(Hs).astype(np.float64)
    else:
        Hs, Hd = H, H.astype(np.float64)
    dtype = tw.TWELL_BF16 if dt == "bf16" else tw.TWELL_F32
    bufs = tw.TwellBuffers(T, F, C, K, dtype)
    tw.twell_pack_dense(torch_dev(Hs), bufs.t)
    code, n = tw.twell_get_status(bufs.t)
    assert code == 0
    g = read(bufs, n)
    ref = oracle.twell_pack(Hd, C, K, dt)
    for k in ("idx", "nnz"):
        assert np.array_equal(g[k], ref[k]), k
    assert np.array_equal(g["val"], ref["val"])
    assert n == ref["n_ovf"] and np.array_equal(g["ovf_rows"], ref["ovf_rows"])
    assert np.array_equal(g["g_fb"], ref["g_fb"])


@pytest.mark.parametrize("hot_every,expect_many", [(100, False), (5, True)])
def test_pack_gate(hot_every, expect_many):
    """Few overflow rows: dense backup rows assembled from slots + wide tiles;
    many (>= 128): recomputed by the tensor-core gate+up GEMM."""
    w = synth.Workload("pk", 640, 256, 1024, 128, 8, "bf16", False, -2.33, 31, hot_tokens=1,
                       seq_len=hot_every, hot_bias=1.6)
    a = synth.generate(w)
    T, D, F = w.T, w.D, w.F
    d = {k: torch_dev(a[k]) for k in ("x", "Wg", "bg", "rb")}
    bufs = tw.TwellBuffers(T, F, w.C, w.K, tw.TWELL_BF16)
    ws, nws = tw.workspace(T, D, F, w.C, w.K, tw.TWELL_BF16, False)
    tw.twell_pack(d["x"], d["Wg"], d["bg"], d["rb"], D, bufs.t, ws, nws)
    code, n = tw.twell_get_status(bufs.t)
    assert code == 0
    assert (n >= 128) == expect_many, n
    g = read(bufs, n)
    z = oracle.gate(a["x"], a["Wg"], a["bg"], a["rb"], "bf16")
    ref = oracle.twell_pack(z, w.C, w.K, "bf16")
    band, _ = z_band(a, "bf16")
    compare_twell(g, ref, z, band, w.C, w.K, "bf16", max_ambiguous=8)
    common = np.intersect1d(g["ovf_rows"], ref["ovf_rows"])
    assert len(common) >= len(ref["ovf_rows"]) - 2
    for t in common:
        gi = int(np.nonzero(g["ovf_rows"] == t)[0][0])
        ri = int(np.nonzero(ref["ovf_rows"] == t)[0][0])
        gr, rr = g["g_fb"][gi], ref["g_fb"][ri]
        assert np.all(np.abs(gr - rr) <= 2.0 ** -7 * np.abs(rr) + 2 * band[t]), t

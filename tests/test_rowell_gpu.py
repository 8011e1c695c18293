"""GPU parity of the row-ELL comparison baseline (classic ELLPACK over the
whole hidden axis): the standalone pack from a dense activation matrix
(bit-exact against the oracle: indices, values, true counts, padding,
capacity status) and the up + down projection that consumes it (against the
oracle within the stated tolerance)."""
import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import oracle
import synth
from twell_testlib import assert_close_rms, to_np64, torch_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    tw.load()


def gate_values(a, dt):
    """g = ReLU(z) in the storage type (the oracle's gate and rounding), as
    the stored bit patterns (bf16) or fp32 values, and as float64."""
    z = oracle.gate(a["x"], a["Wg"], a["bg"], a["rb"], dt)
    z32 = z.astype(np.float32)
    g32 = np.where(z32 > 0, z32, np.float32(0))
    if dt == "bf16":
        bits = oracle.bf16_round(g32)
        g = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return bits, g
    return g32, g32.astype(np.float64)


def run_rowell(a, w, E):
    dt = w.dtype
    dtype = tw.TWELL_BF16 if dt == "bf16" else tw.TWELL_F32
    store, g = gate_values(a, dt)
    re = tw.RowEllBuffers(w.T, w.F, E, dtype)
    tw.twell_rowell_pack_dense(torch_dev(store), re.t)
    d = {k: torch_dev(a[k]) for k in ("x", "Wu", "Wd")}
    y = torch.full((w.T, w.D), float("nan"), dtype=torch.bfloat16 if dt == "bf16" else torch.float32,
                   device="cuda")
    tw.twell_rowell_forward(d["x"], d["Wu"], d["Wd"], w.D, re.t, y)
    torch.cuda.synchronize()
    return re, g, to_np64(y)


@pytest.mark.parametrize("dt,gated,D", [("bf16", True, 256), ("bf16", False, 200),
                                        ("f32", True, 128), ("bf16", True, 2048)])
def test_rowell_pack_and_forward(dt, gated, D):
    w = synth.Workload(f"re{dt}{D}", 300, D, 1024, 128, 8, dt, gated, -2.0, 60 + D % 97,
                       hot_tokens=3, seq_len=100, hot_bias=1.4)
    a = synth.generate(w)
    _, g = gate_values(a, dt)
    E = int((g > 0).sum(axis=1).max())  # the densest row sets the width
    re, g, y = run_rowell(a, w, E)
    ref = oracle.rowell_pack(g, E)
    assert int(re.status[0].item()) == 0
    assert np.array_equal(re.nnz.cpu().numpy(), ref["nnz"])
    assert np.array_equal(re.idx.cpu().numpy().view(np.uint16), ref["idx"])
    assert np.array_equal(to_np64(re.val), ref["val"])
    y_ref = oracle.ffn_rowell(a["x"], a["Wu"], a["Wd"], ref, dt)
    assert_close_rms(y, y_ref, dt, "y")
    # and the FFN it computes is the dense FFN of the oracle
    y_dense = oracle.ffn_dense(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], dt, dt)
    assert np.array_equal(y_ref, y_dense)


def test_rowell_capacity_status_and_first_entries():
    w = synth.Workload("recap", 200, 128, 512, 128, 8, "bf16", True, -1.5, 71)
    a = synth.generate(w)
    _, g = gate_values(a, "bf16")
    E = 8
    assert (g > 0).sum(axis=1).max() > E
    re, g, _ = run_rowell(a, w, E)
    assert int(re.status[0].item()) == -4  # TWELL_ERR_CAPACITY
    ref = oracle.rowell_pack(g, E)
    assert np.array_equal(re.nnz.cpu().numpy(), ref["nnz"])
    assert np.array_equal(re.idx.cpu().numpy().view(np.uint16), ref["idx"])
    assert np.array_equal(to_np64(re.val), ref["val"])


def test_rowell_rejects_bad_arguments():
    re = tw.RowEllBuffers(64, 100, 4, tw.TWELL_BF16)  # F not a multiple of 32
    with pytest.raises(tw.TwellError):
        tw.twell_rowell_pack_dense(torch.zeros((64, 100), dtype=torch.bfloat16, device="cuda"), re.t)

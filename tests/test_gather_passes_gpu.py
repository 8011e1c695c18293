"""The gather kernels split into passes (twell_t.gather_passes): the forward's
up projection and down projection as two passes with h at the slots in
between, and the backward's dx and weight-gradient gathers over column
ranges of d_model.  Every output element sums the same products in the
same order whatever the pass count, so the results must be bit-identical to
the single-pass run; the split runs are also checked against the oracle."""
import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import oracle
import synth
from twell_testlib import assert_close_rms, check_backward, run_train, value_allowance

pytestmark = pytest.mark.gpu

OUTS = ("y", "dx", "dWg", "dWu", "dWd", "dbg")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    tw.load()


def same(g1, g2):
    for k in OUTS:
        if g1[k] is None:
            assert g2[k] is None
            continue
        assert np.array_equal(g1[k], g2[k]), k


CASES = {
    # bf16 gated, a few overflow rows on the gathers (wide tiles / backup rows)
    "bf16_gated_ovf": synth.Workload("gp1", 300, 2048, 1024, 128, 8, "bf16", True, -2.33, 61,
                                     hot_tokens=3, seq_len=100, hot_bias=1.49, train=True),
    # d_model 1024 (128 vectors: three passes of 42 / 43 / 43), ragged T
    "bf16_d1024": synth.Workload("gp2", 257, 1024, 512, 64, 4, "bf16", True, -1.9, 62,
                                 train=True),
    # fp32 (4-element vectors), gated
    "f32_gated": synth.Workload("gp3", 130, 512, 512, 64, 8, "f32", True, -1.7, 63, train=True),
    # plain FFN: no up pass; dx / dW still split
    "bf16_plain": synth.Workload("gp4", 200, 1024, 512, 128, 8, "bf16", False, -1.8, 64,
                                 hot_tokens=2, seq_len=100, hot_bias=1.5, train=True),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("passes", [2, 3, 4])
def test_passes_bit_identical(case, passes):
    w = CASES[case]
    a = synth.generate(w)
    g1 = run_train(a, w, 1e-3, gather_passes=1)
    gp = run_train(a, w, 1e-3, gather_passes=passes)
    assert g1["code"] == 0 and gp["code"] == 0
    same(g1, gp)


@pytest.mark.parametrize("case", ["bf16_gated_ovf", "f32_gated"])
def test_split_passes_match_the_oracle(case):
    w = CASES[case]
    a = synth.generate(w)
    g = run_train(a, w, 1e-3, gather_passes=2)
    assert g["code"] == 0
    y_ref = oracle.ffn_dense(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], w.dtype, w.dtype)
    extra = value_allowance(a, w.dtype, want=("y",))["y"]
    assert_close_rms(g["y"], y_ref, w.dtype, "y", extra=extra)
    check_backward(a, w, g, 1e-3)


def test_more_passes_than_vectors():
    """d_model 64 bf16 is 8 vectors per row: a request for more passes than
    that is clamped (one vector per pass) and still bit-identical."""
    w = synth.Workload("gp5", 96, 64, 256, 64, 4, "bf16", True, -1.5, 65, train=True)
    a = synth.generate(w)
    g1 = run_train(a, w, 1e-3, gather_passes=1)
    g9 = run_train(a, w, 1e-3, gather_passes=64)
    assert g1["code"] == 0 and g9["code"] == 0
    same(g1, g9)


def test_config4_shape_default_equals_one_pass():
    """d_model 4096 / d_ff 14336 (the shape where the library splits by
    default), fewer tokens: the default run equals a forced single pass."""
    w = synth.Workload("gp6", 512, 4096, 14336, 128, 8, "bf16", True, -2.58, 66, train=True)
    a = synth.generate(w)
    g0 = run_train(a, w, 1e-4, gather_passes=0)
    g1 = run_train(a, w, 1e-4, gather_passes=1)
    assert g0["code"] == 0 and g1["code"] == 0
    same(g0, g1)

"""Pins of the row-ELL comparison oracle (classic ELLPACK over the whole
hidden axis, the format the technical summary's section 2.A contrasts TwELL
with): a hand-worked case, the inverse of the pack, agreement with the
independently pinned TwELL pack on rows that fit their slots, the capacity
rule, and the FFN identity (row-ELL FFN == dense FFN, bit-exact)."""
import numpy as np
import pytest

import oracle
from test_oracle import active_np, q_np, small_case


def test_rowell_hand_worked_case():
    h = np.array([[0, 1.5, 0, 2, 0, 0, 3, 0],
                  [0, 0, 0, 0, 0, 0, 0, 0],
                  [4, 0, 0, 0, 0, 0, 0, 5]], dtype=np.float64)
    r = oracle.rowell_pack(h, 2)
    assert r["idx"].tolist() == [[1, 3], [0xFFFF, 0xFFFF], [0, 7]]
    assert r["val"].tolist() == [[1.5, 2.0], [0.0, 0.0], [4.0, 5.0]]
    assert r["nnz"].tolist() == [3, 0, 2]  # the true count, past the width


@pytest.mark.parametrize("seed", [0, 1])
def test_rowell_unpack_is_identity(seed):
    rng = np.random.default_rng(seed)
    h = np.maximum(rng.standard_normal((37, 96)) - 1.5, 0.0)
    E = int((h > 0).sum(axis=1).max())
    r = oracle.rowell_pack(h, E)
    back = np.zeros_like(h)
    for t in range(h.shape[0]):
        m = r["nnz"][t]
        assert np.all(np.diff(r["idx"][t, :m].astype(np.int64)) > 0)  # ascending
        assert np.all(r["idx"][t, m:] == 0xFFFF) and np.all(r["val"][t, m:] == 0)
        back[t, r["idx"][t, :m]] = r["val"][t, :m]
    assert np.array_equal(back, h)


def test_rowell_capacity_keeps_first_entries():
    rng = np.random.default_rng(3)
    h = np.maximum(rng.standard_normal((20, 64)), 0.0)
    full = oracle.rowell_pack(h, 64)
    short = oracle.rowell_pack(h, 5)
    assert np.array_equal(short["nnz"], full["nnz"])
    assert np.array_equal(short["idx"], full["idx"][:, :5])
    assert np.array_equal(short["val"], full["val"][:, :5])


@pytest.mark.parametrize("C,K", [(8, 2), (32, 8)])
def test_rowell_agrees_with_twell_on_fitting_rows(C, K):
    """On a row whose tiles all fit their K slots, the row-ELL entries are the
    TwELL slots of its tiles in tile order, with global columns j*C + idx."""
    a = small_case(23, 32, 64, "bf16", True, 31, -1.2, hot=np.where(np.arange(23) < 3, 1.5, 0.0))
    z = oracle.gate(a["x"], a["Wg"], a["bg"], a["rb"], "bf16")
    tw = oracle.twell_pack(z, C, K, "bf16")
    g = np.where(active_np(z, "bf16"), q_np(z, "bf16"), 0.0)
    re = oracle.rowell_pack(g, 64)
    fitting = [t for t in range(23) if not tw["row_ovf"][t]]
    assert len(fitting) > 5
    for t in fitting:
        cols, vals = [], []
        for j in range(64 // C):
            n = tw["nnz"][j, t]
            cols += [j * C + int(c) for c in tw["idx"][j, t, :n]]
            vals += list(tw["val"][j, t, :n])
        m = re["nnz"][t]
        assert m == len(cols)
        assert re["idx"][t, :m].tolist() == cols and re["val"][t, :m].tolist() == vals


@pytest.mark.parametrize("dt,gated,q", [("bf16", True, "bf16"), ("f32", False, "f32")])
def test_rowell_ffn_equals_dense_bit_exact(dt, gated, q):
    """The FFN over row-ELL gate values reproduces the dense FFN exactly (the
    dense loop adds only h = 0 terms, in the same ascending order)."""
    a = small_case(23, 32, 64, dt, gated, 41, -1.0, hot=np.where(np.arange(23) < 2, 1.5, 0.0))
    z = oracle.gate(a["x"], a["Wg"], a["bg"], a["rb"], dt)
    g = np.where(active_np(z, q), q_np(z, q), 0.0)
    re = oracle.rowell_pack(g, int((g > 0).sum(axis=1).max()))
    y_re = oracle.ffn_rowell(a["x"], a["Wu"], a["Wd"], re, dt)
    y_de = oracle.ffn_dense(a["x"], a["Wg"], a["bg"], a["rb"], a["Wu"], a["Wd"], dt, q)
    assert np.array_equal(y_re, y_de) and np.abs(y_de).max() > 0

"""The allocation-free hybrid split, for callers that cannot allocate device
memory (code inside an allocator or pool it does not own, hosts that forbid
allocation on their hot path).  twell_hybrid_split_static keeps its scratch in
a fixed device array inside the library; its overflow-row list must equal the
one the workspace-free packing entry point (twell_pack_dense) produces for
the same activations, and the oracle's list from the same activations, on
consecutive calls that share that array.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import oracle
import synth
from twell_testlib import torch_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    lib = tw.load()
    lib.twell_hybrid_split_static.argtypes = [ctypes.POINTER(tw.twell_t), ctypes.c_void_p]
    lib.twell_hybrid_split_static.restype = ctypes.c_int
    return lib


def activations(T, F, seed, hot_every):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((T, F)).astype(np.float32)
    p = np.where(np.arange(T) % hot_every == 0, 0.3, 0.01)[:, None]
    H = np.where(rng.random((T, F)) < p, np.abs(H), 0.0).astype(np.float32)
    return synth.f32_to_bf16_bits(H)


def packed(H, C, K, cap=None):
    """TwELL + overflow list from the existing entry point."""
    T, F = H.shape
    a = tw.TwellBuffers(T, F, C, K, tw.TWELL_BF16, ovf_cap=cap)
    tw.twell_pack_dense(torch_dev(H), a.t)
    code, n = tw.twell_get_status(a.t)
    return a, code, n


def split_static(lib, a, cap=None):
    """Same TwELL counts, list recomputed by the allocation-free entry point."""
    T, F, C, K = a.T, a.F, a.C, a.K
    b = tw.TwellBuffers(T, F, C, K, tw.TWELL_BF16, ovf_cap=cap)
    b.nnz.copy_(a.nnz)
    b.ovf_rows.fill_(-7)
    b.n_ovf.fill_(-1)
    code = lib.twell_hybrid_split_static(ctypes.byref(b.t),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, code
    st, n = tw.twell_get_status(b.t)
    return b, st, n


def oracle_list(H, C, K):
    """Overflow rows of H by the oracle's TwELL pack (active iff > 0)."""
    ref = oracle.twell_pack(synth.to_f64(H, "bf16"), C, K, "bf16")
    return ref["ovf_rows"]


def test_matches_existing_entry_on_two_calls_in_a_row(lib):
    T, F, C, K = 3000, 1024, 128, 8
    for seed, hot in ((1, 37), (2, 5)):          # different overflow sets, same array
        H = activations(T, F, seed, hot)
        a, code_a, n_a = packed(H, C, K)
        b, code_b, n_b = split_static(lib, a)
        assert code_a == 0 and code_b == 0
        assert n_a > 0 and n_b == n_a
        assert torch.equal(b.ovf_rows[:n_b], a.ovf_rows[:n_a])
        want = oracle_list(H, C, K)
        assert n_b == len(want)
        assert np.array_equal(b.ovf_rows[:n_b].cpu().numpy(), want)


def test_capacity_and_static_limit(lib):
    T, F, C, K = 700, 512, 64, 4
    H = activations(T, F, 3, 3)
    a, _, n_a = packed(H, C, K)
    b, st, n_b = split_static(lib, a, cap=5)
    assert n_b == n_a > 5
    assert st == -4                                 # TWELL_ERR_CAPACITY on the device
    assert torch.equal(b.ovf_rows[:5], a.ovf_rows[:5])
    assert np.array_equal(b.ovf_rows[:5].cpu().numpy(), oracle_list(H, C, K)[:5])
    # more tokens than the fixed scratch holds: rejected before any launch
    big = tw.twell_t(T=262145, F=512, C=64, K=4, dtype=tw.TWELL_BF16, idx=1 << 40, val=1 << 40,
                     nnz=1 << 40, ovf_rows=1 << 40, n_ovf=1 << 40, ovf_cap=1, g_fb=1 << 40,
                     u_val=None, u_fb=None, status=1 << 40, dense_switch=0.0)
    assert lib.twell_hybrid_split_static(ctypes.byref(big), None) == -10

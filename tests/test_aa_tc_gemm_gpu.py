"""The tcgen05 GEMM engine through its test hook (the test-hooks build of the
library), on exact integer inputs
(every fp32 accumulation order gives the same value), then on Gaussian
inputs.  Runs first among the GPU tests: the TwELL kernels sit on this engine."""
import ctypes

import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hook():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build(variants=("hooks",))
    lib = tw.load(tw._build.lib_path("hooks"))
    f = lib.twell_test_tc_gemm
    P = ctypes.c_void_p
    f.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
    f.restype = ctypes.c_int
    return f


def run(hook, A, B, M, N, K, layout):
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    code = hook(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, layout, st.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
    assert code == 0, code
    torch.cuda.synchronize()
    assert int(st[0]) == 0, f"device status {int(st[0])}"
    return C.cpu().numpy().astype(np.float64)


def describe_mismatch(got, want):
    bad = got != want
    rows = np.nonzero(bad.any(axis=1))[0]
    cols = np.nonzero(bad.any(axis=0))[0]
    return (f"{int(bad.sum())} of {bad.size} differ; rows {rows[:8].tolist()}.. ({len(rows)}), "
            f"cols {cols[:8].tolist()}.. ({len(cols)}); got[0,:4]={got[0, :4]} want={want[0, :4]}")


def operands(g, M, N, K, layout, draw):
    """A, B in the storage the layout names (bit 0: B [K][N], bit 1: A [K][M])
    and the float64 product C = op(A) op(B)."""
    A = draw((K, M) if layout & 2 else (M, K), g).to(torch.bfloat16)
    B = draw((K, N) if layout & 1 else (N, K), g).to(torch.bfloat16)
    a = A.double().numpy()
    b = B.double().numpy()
    a = a.T if layout & 2 else a
    b = b if layout & 1 else b.T
    return A, B, a, b


@pytest.mark.parametrize("M,N,K,layout", [
    (128, 128, 64, 0), (256, 256, 256, 0), (200, 384, 320, 0), (77, 136, 72, 0),
    (128, 128, 64, 1), (256, 256, 256, 1), (300, 192, 512, 1), (64, 72, 200, 1),
    (128, 128, 64, 2), (256, 136, 192, 2), (200, 256, 72, 3), (384, 264, 300, 3),
])
def test_tc_gemm_integer_exact(hook, M, N, K, layout):
    """layout 2, 3: A read MN-major (the weight-gradient GEMMs of the backward),
    with ragged M and a K that is not a multiple of the 64-deep k-block."""
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K + layout)
    A, B, a, b = operands(g, M, N, K, layout, lambda sh, gg: torch.randint(-3, 4, sh, generator=gg))
    want = a @ b
    got = run(hook, A.cuda(), B.cuda(), M, N, K, layout)
    assert np.array_equal(got, want), describe_mismatch(got, want)


@pytest.mark.parametrize("layout", [0, 1, 2, 3])
def test_tc_gemm_gaussian(hook, layout):
    M, N, K = 512, 640, 1024
    g = torch.Generator().manual_seed(5 + layout)
    A, B, a, b = operands(g, M, N, K, layout, lambda sh, gg: torch.randn(sh, generator=gg))
    want = a @ b
    bound = K * 2.0 ** -23 * (np.abs(a) @ np.abs(b))
    got = run(hook, A.cuda(), B.cuda(), M, N, K, layout)
    assert np.all(np.abs(got - want) <= bound)

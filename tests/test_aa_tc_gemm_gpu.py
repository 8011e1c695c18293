"""The tcgen05 GEMM engine through its test hook, on exact integer inputs
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
    tw._build.build()
    lib = tw.load()
    f = lib.twell_test_tc_gemm
    P = ctypes.c_void_p
    f.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
    f.restype = ctypes.c_int
    return f


def run(hook, A, B, M, N, K, b_mn):
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    code = hook(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, b_mn, st.data_ptr(),
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


@pytest.mark.parametrize("M,N,K,b_mn", [
    (128, 128, 64, 0), (256, 256, 256, 0), (200, 384, 320, 0), (77, 136, 72, 0),
    (128, 128, 64, 1), (256, 256, 256, 1), (300, 192, 512, 1), (64, 72, 200, 1),
])
def test_tc_gemm_integer_exact(hook, M, N, K, b_mn):
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K + b_mn)
    A = torch.randint(-3, 4, (M, K), generator=g).to(torch.bfloat16)
    if b_mn:
        B = torch.randint(-3, 4, (K, N), generator=g).to(torch.bfloat16)
        want = A.double().numpy() @ B.double().numpy()
    else:
        B = torch.randint(-3, 4, (N, K), generator=g).to(torch.bfloat16)
        want = A.double().numpy() @ B.double().numpy().T
    got = run(hook, A.cuda(), B.cuda(), M, N, K, b_mn)
    assert np.array_equal(got, want), describe_mismatch(got, want)


@pytest.mark.parametrize("b_mn", [0, 1])
def test_tc_gemm_gaussian(hook, b_mn):
    M, N, K = 512, 640, 1024
    g = torch.Generator().manual_seed(5 + b_mn)
    A = torch.randn((M, K), generator=g).to(torch.bfloat16)
    B = torch.randn((K, N) if b_mn else (N, K), generator=g).to(torch.bfloat16)
    a, b = A.double().numpy(), B.double().numpy()
    want = a @ b if b_mn else a @ b.T
    bound = K * 2.0 ** -23 * (np.abs(a) @ (np.abs(b) if b_mn else np.abs(b).T))
    got = run(hook, A.cuda(), B.cuda(), M, N, K, b_mn)
    assert np.all(np.abs(got - want) <= bound)

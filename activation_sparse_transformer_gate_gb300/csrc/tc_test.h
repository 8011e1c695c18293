// tc_test.h -- test hook of the tcgen05 GEMM engine (exported, not part of the
// public ABI in include/twell.h): fp32 C[M][N] = A[M][K] B^T with B [N][K]
// (b_mn = 0) or A B with B [K][N] (b_mn = 1); A, B bf16 device pointers,
// K % 8 == 0 (16-byte row pitch), N % 8 == 0 when b_mn = 1.  Returns a
// twell_status code; device-side errors go to *status.
#pragma once
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif
int twell_test_tc_gemm(const void *A, const void *B, float *C, int M, int N, int K, int b_mn,
                       int32_t *status, void *stream);
#ifdef __cplusplus
}
#endif

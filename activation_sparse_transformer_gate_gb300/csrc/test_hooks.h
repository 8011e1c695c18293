// test_hooks.h -- test and measurement hooks, compiled only into the
// test-hooks variant of the library (TWELL_TEST_HOOKS), never into
// libtwell.so, and not part of the public ABI in include/twell.h.
//
// twell_test_tc_gemm: the tcgen05 GEMM engine with a plain fp32 epilogue,
// C[M][N] = op(A) op(B), A and B bf16 device pointers.  layout bit 0: B is
// [K][N] (MN-major), else [N][K]; bit 1: A is [K][M] (MN-major), else
// [M][K].  Every row pitch must be a multiple of 16 bytes (the inner extent
// a multiple of 8).  Returns a twell_status code; device-side errors go to
// *status.
//
// twell_test_gather_probe: gather n_rows rows (indices in rows[], each < the
// row count of W, checked by the caller) of row_bytes each from W with
// `blocks` CTAs of 256 threads; out receives blocks * 8 checksums.
// Asynchronous on stream.
#pragma once
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif
int twell_test_tc_gemm(const void *A, const void *B, float *C, int M, int N, int K, int layout,
                       int32_t *status, void *stream);
int twell_test_gather_probe(const void *W, int row_bytes, const int32_t *rows, int n_rows,
                            int blocks, uint32_t *out, void *stream);
#ifdef __cplusplus
}
#endif

// probe.cu -- measurement hook, compiled only into the test-hooks variant of
// the library (not into libtwell.so; not part of the public ABI in
// include/twell.h): the rate at which this GPU gathers rows of a matrix in
// an arbitrary order, the access pattern of the sparse projections.  Warps
// take consecutive entries of a row list; every lane loads its 16-byte
// vectors of each row (read-only, no L1 allocation, evict-normal in L2) and
// folds them into a checksum, so the loads cannot be elided.  The result is
// the memory system's ceiling for the gathers (mostly L2 hits when the matrix
// fits in L2), against which the gather kernels can be read.
#include "common.cuh"
#include "kernels.h"
#include "test_hooks.h"

namespace twell {

namespace {

constexpr int PROBE_THREADS = 256;

__global__ void __launch_bounds__(PROBE_THREADS) gather_probe_kernel(
    const uint4 *__restrict__ W, int row_vecs, const int32_t *__restrict__ rows, int n_rows,
    int per_warp, uint32_t *__restrict__ out) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const long j0 = (long)gw * per_warp;
  const long j1 = j0 + per_warp < n_rows ? j0 + per_warp : n_rows;
  uint32_t acc = 0;
  for (long j = j0; j < j1; ++j) {
    const uint4 *row = W + (size_t)rows[j] * row_vecs;
    for (int v = lane; v < row_vecs; v += 32) {
      const uint4 r = ldg_stream(row + v);
      acc ^= r.x ^ r.y ^ r.z ^ r.w;
    }
  }
  out[gw] = acc;
}

}  // namespace

}  // namespace twell

// W: [n_mat][row_bytes] device matrix; rows: n_rows indices in [0, n_mat)
// (checked by the caller); out: one uint32 per warp of the launch, i.e.
// blocks * 8 entries.  row_bytes a positive multiple of 16.
extern "C" int twell_test_gather_probe(const void *W, int row_bytes, const int32_t *rows,
                                       int n_rows, int blocks, uint32_t *out, void *stream) {
  using namespace twell;
  if (!W || !rows || !out || row_bytes <= 0 || (row_bytes % 16) || n_rows < 1 || blocks < 1)
    return TWELL_ERR_ARG;
  const int warps = blocks * (PROBE_THREADS / 32);
  const int per_warp = (n_rows + warps - 1) / warps;
  gather_probe_kernel<<<blocks, PROBE_THREADS, 0, (cudaStream_t)stream>>>(
      (const uint4 *)W, row_bytes / 16, rows, n_rows, per_warp, out);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

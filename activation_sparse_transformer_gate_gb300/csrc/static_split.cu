// static_split.cu -- the hybrid split (overflow-row list of a packed TwELL)
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a memory
// pool or arena they do not own, plugin hosts that forbid allocation on their
// hot path, or processes that have handed all device memory to another
// allocator.  For them this entry point keeps its scratch (the overflow-row
// bitmap, the full row list, per-row positions and the control block that the
// workspace-based split uses) in one file-scope device array of fixed size,
// so a call needs nothing but the caller's TwELL buffers.
//
// The array lives in the library image: every GPU that loads the library
// holds it (about 2 MiB) until the process exits.  All calls share it and it
// keeps the previous call's contents; the bitmap is cleared at the start of
// every call.  Calls that overlap on the GPU (different streams, or different
// host threads on the same device without ordering) race on it.
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace twell {

namespace {

constexpr int kMaxT = TWELL_STATIC_SPLIT_MAX_T;
constexpr size_t kCtlBytes = 256;
constexpr size_t kBitsBytes = ((size_t)kMaxT / 32) * 4;
constexpr size_t kRowsBytes = (size_t)kMaxT * 4;
constexpr size_t kScratchBytes = kCtlBytes + kBitsBytes + 2 * kRowsBytes;
static_assert(kMaxT % 32 == 0 && kBitsBytes % 256 == 0 && kRowsBytes % 256 == 0,
              "scratch regions must stay 256-byte aligned");

// Host code may only use the name of this array through cudaGetSymbolAddress:
// on the host it is a stand-in, not a device address.
static __device__ __align__(256) unsigned char g_split_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char *g_ptr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once per
// device, with that device current).
cudaError_t scratch_ptr(unsigned char **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = (unsigned char *)p;
  }
  *out = g_ptr[dev];
  return cudaSuccess;
}

bool ok_ck(int C, int K) {
  const bool k2 = K == 1 || K == 2 || K == 4 || K == 8 || K == 16 || K == 32;
  return (C == 32 || C == 64 || C == 128) && k2 && K <= C;
}

}  // namespace

}  // namespace twell

using namespace twell;

extern "C" twell_status twell_hybrid_split_static(twell_t *tw, void *stream) {
  if (!tw) return TWELL_ERR_ARG;
  if (tw->T < 1 || tw->F < 1 || !ok_ck(tw->C, tw->K) || tw->F % tw->C != 0) return TWELL_ERR_ARG;
  if (tw->T > kMaxT) return TWELL_ERR_STATIC_LIMIT;
  if ((double)tw->T * (double)(tw->F / tw->C) * (double)tw->K >= 2147483647.0) return TWELL_ERR_ARG;
  if (!tw->nnz || !tw->n_ovf || !tw->status || tw->ovf_cap < 0) return TWELL_ERR_ARG;
  if (tw->ovf_cap > 0 && !tw->ovf_rows) return TWELL_ERR_ARG;
  unsigned char *base = nullptr;
  if (scratch_ptr(&base) != cudaSuccess) return TWELL_ERR_CUDA;
  Workspace ws;
  memset(&ws, 0, sizeof(ws));
  ws.ctl = (Ctl *)base;
  ws.ovf_bits = (uint32_t *)(base + kCtlBytes);
  ws.rows = (int32_t *)(base + kCtlBytes + kBitsBytes);
  ws.pos = (int32_t *)(base + kCtlBytes + kBitsBytes + kRowsBytes);
  cudaStream_t s = (cudaStream_t)stream;
  // the bit of every row with a tile over K (every bitmap word written)
  cudaError_t e = launch_flags_from_nnz(*tw, ws.ovf_bits, nullptr, s);
  if (e == cudaSuccess) e = launch_overflow_compact(*tw, &ws, 2.0f, s, /*write_user=*/true);
  return e == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

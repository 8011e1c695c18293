// static_split.cu -- the hybrid split (overflow-row list of a packed TwELL)
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a memory
// pool or arena they do not own, plugin hosts that forbid allocation on their
// hot path, or processes that have handed all device memory to another
// allocator.  For them this entry point keeps its scratch (the overflow-row
// bitmap, the full row list, per-row positions and the control block that the
// workspace-based split uses) in one file-scope device array of fixed size,
// so a call needs nothing but the caller's TwELL buffers: it makes no
// cudaMalloc or cudaFree call and uses no allocating library routine.
//
// The array lives in the library image: every GPU that loads the library
// holds it (about 2 MiB) until the process exits.  All calls share it and it
// keeps the previous call's contents; the bitmap is cleared at the start of
// every call.  Calls that overlap on the GPU (different streams, or different
// host threads on the same device without ordering) race on it.
#include <cuda.h>
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

// The array's address belongs to a CUDA context: a device reset (or another
// context on the same device) gives the array another address.  The address
// is therefore looked up once per context, identified by the driver's
// process-unique context id (a context handle may be reused after a reset;
// its id is not), with that context current, and cached.
constexpr int kMaxContexts = 64;
struct CtxAddr {
  unsigned long long ctx_id;
  unsigned char *ptr;
};
std::mutex g_mu;
CtxAddr g_addr[kMaxContexts] = {};
int g_n_addr = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <class Fn>
Fn driver_fn(const char *name) {
  void *f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return (Fn)f;
}

// Id of the current context.  The runtime creates its context lazily: when
// none is current yet, the symbol lookup (which needs one) creates it first.
cudaError_t current_ctx_id(unsigned long long *id) {
  static CtxGetCurrentFn get_cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_cur || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (!ctx) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) return e;
    if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorUnknown;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// Device address of the array in the current context (looked up with that
// context current on the first call in it).
cudaError_t scratch_ptr(unsigned char **out) {
  unsigned long long id = 0;
  cudaError_t e = current_ctx_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(g_mu);
  for (int i = 0; i < g_n_addr; ++i)
    if (g_addr[i].ctx_id == id) {
      *out = g_addr[i].ptr;
      return cudaSuccess;
    }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_split_scratch);
  if (e != cudaSuccess) return e;
  // keep the most recent contexts (a process rarely has more than one per device)
  const int slot = g_n_addr < kMaxContexts ? g_n_addr++ : (int)(id % kMaxContexts);
  g_addr[slot] = {id, (unsigned char *)p};
  *out = (unsigned char *)p;
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

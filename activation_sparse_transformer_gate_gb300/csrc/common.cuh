// common.cuh -- device helpers shared by the TwELL kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "twell.h"

namespace twell {

using bf16 = __nv_bfloat16;

// ---- element conversions ---------------------------------------------------
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }

template <class T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// bf16 pair packed in a 32-bit word -> two floats (exact widening).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> bf16 pair (round to nearest even), low half = a.
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&p);
}

// Bit pattern of the storage value of v (for assembling vector stores).
__device__ __forceinline__ uint32_t store_bits(float v, float *) { return __float_as_uint(v); }
__device__ __forceinline__ uint32_t store_bits(float v, bf16 *) {
  bf16 b = __float2bfloat16_rn(v);
  return (uint32_t)(*reinterpret_cast<uint16_t *>(&b));
}

// L2 cache policy of gathered rows.  A read-only load that skips L1 otherwise
// enters L2 with evict-first priority, and a gathered weight row is read again
// by many other tokens: with evict-first the weight matrices miss L2 although
// they fit in it.  L2_FIRST keeps that priority for rows read once.
// (Pure asm: the compiler may hoist and share it.)
enum L2Pol { L2_NORMAL = 0, L2_FIRST = 1 };

template <int POL>
__device__ __forceinline__ uint64_t gather_policy() {
  uint64_t pol;
  if (POL == L2_FIRST)
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  else
    asm("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 16-byte read-only load of a gathered row: no L1 allocation, L2 policy POL.
template <int POL = L2_NORMAL>
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(gather_policy<POL>()));
  return r;
}

// 32-byte read-only load (two 16-byte vectors; the address must be 32-byte
// aligned): no L1 allocation, L2 policy POL.
template <int POL = L2_NORMAL>
__device__ __forceinline__ void ldg_stream32(const void *p, uint4 &a, uint4 &b) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
      : "l"(p), "l"(gather_policy<POL>()));
}

// 16-byte store of a row that is not read again by the same kernel (y, dx,
// dW rows): no L1 allocation, evict-first in L2, so the stream of outputs
// does not displace the gathered weight rows.
__device__ __forceinline__ void stg_stream(void *p, const uint4 &v) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
               ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(gather_policy<L2_FIRST>())
               : "memory");
}

// ---- programmatic dependent launch -------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialization, and each kernel's first statement is pdl_begin(), which
// waits until the previous kernel of the stream has completed and its memory
// is visible (nothing is read or written before it).  The kernels do not
// trigger their dependents early, so a dependent is scheduled as the previous
// grid's last CTAs exit: the overlap covers launch latency only, and at most
// two grids are in flight.  That hides most of the launch gap between the
// short, dependent kernels of a step (several of which exit at once when the
// dispatcher chose no work for them): the training step at T=4096,
// d_model 2048, d_ff 8192 went from 0.907 to 0.869 ms.  (Triggering
// dependents at the start of every CTA let chains of idle kernels all be in
// flight at once and made the same step 0.965 ms.)
// TWELL_PDL=0 in the environment launches plainly.
__device__ __forceinline__ void pdl_begin() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

inline bool pdl_enabled() {
  static const bool on = [] {
    const char *e = getenv("TWELL_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---- device status word ------------------------------------------------------
__device__ __forceinline__ void set_status(int32_t *st, int code) {
  if (st) atomicCAS(st, 0, code);
}

// ---- control block in the workspace -----------------------------------------
// Written by the overflow-compaction kernel, read by everything after it.
// Overflow rows go through the tensor-core dense-row GEMMs when there are at
// least this many of them (one full M tile); fewer go through the gather
// kernels, which read their overflowing tiles from the wide-tile buffer.
constexpr int OVF_GEMM_MIN = 128;

struct Ctl {
  int32_t n_rows;   // rows on the dense GEMM path: T (all-dense), n_ovf (ovf_gemm) or 0
  int32_t dense;    // 1: every row runs densely (n_ovf > dense_switch * T, or dense slots)
  int32_t n_ovf;    // true number of overflow rows
  int32_t ovf_gemm; // 1: overflow rows run on the dense GEMM path
  unsigned long long slots;  // TwELL slots written by the gate epilogue (zeroed before it)
  int32_t dh_gemm;  // backward: dh of the sparse rows from one dense GEMM read at the slots
  int32_t pad[9];
};

}  // namespace twell

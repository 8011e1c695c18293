// rowell.cu -- classic row-ELL, the comparison baseline for TwELL.
//
// "Sparser, Faster, Lighter Transformer Language Models", technical summary
// section 2.A contrasts TwELL with ELLPACK: one list of (column, value)
// entries per row over the whole hidden axis, padded to a common width E, so
// the width is set by the densest row and the format cannot be written in a
// GEMM epilogue (a row spans every N-tile of the output).  Here it is built
// the only way it can be: the gate matmul writes the dense activation matrix
// H, and a standalone pass packs it.  The up + down projection that consumes
// it gathers the same W_up / W_down rows as the TwELL kernel, so the two
// formats differ in what the comparison is about: packing (fused epilogue
// against a pass over H) and width (per-tile K against the densest row).
//
// Layout: idx [T][E] uint16 global column, ascending, pad 0xFFFF; val [T][E]
// (dtype), pad +0; nnz [T] int32, the true count (may exceed E: the entries
// past E are dropped and the status word gets TWELL_ERR_CAPACITY).
#include "common.cuh"
#include "gather.cuh"
#include "kernels.h"

namespace twell {

namespace {

constexpr int RE_THREADS = 128;  // up + down: one CTA of four warps per token
constexpr int RE_CHUNK = 1024;   // entries staged in shared memory at a time

// One warp per row: each lane tests a 16-byte vector of H (8 bf16 / 4 fp32
// values), a warp scan of the per-lane counts gives each positive value its
// position, entries are written in ascending column order.
template <class T>
__global__ void __launch_bounds__(256)
    rowell_pack_dense_kernel(const T *__restrict__ H, int Tn, int F, int E,
                             uint16_t *__restrict__ idx, T *__restrict__ val,
                             int32_t *__restrict__ nnz, int32_t *status) {
  pdl_begin();
  constexpr int EV = Vec<T>::EV;
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int NV = F / EV;  // F is a multiple of 32
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < Tn; t += gridDim.x * warps) {
    const uint4 *row = (const uint4 *)(H + (size_t)t * F);
    uint16_t *ri = idx + (size_t)t * E;
    T *rv = val + (size_t)t * E;
    int base = 0;
    for (int v0 = 0; v0 < NV; v0 += 32) {
      const int vi = v0 + lane;
      float f[EV];
      const uint4 w = vi < NV ? ldg_stream<L2_FIRST>(row + vi) : make_uint4(0, 0, 0, 0);
      Vec<T>::unpack(w, f);
      unsigned lm = 0;
#pragma unroll
      for (int e = 0; e < EV; ++e) lm |= (f[e] > 0.f ? 1u : 0u) << e;
      const int cnt = __popc(lm);
      int inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      int pos = base + inc - cnt;
#pragma unroll
      for (int e = 0; e < EV; ++e) {
        if ((lm >> e) & 1u) {
          if (pos < E) {
            ri[pos] = (uint16_t)(vi * EV + e);
            rv[pos] = from_f<T>(f[e]);
          }
          ++pos;
        }
      }
      base += __shfl_sync(0xffffffffu, inc, 31);
    }
    for (int k = base + lane; k < E; k += 32) {
      ri[k] = 0xFFFFu;
      rv[k] = from_f<T>(0.f);
    }
    if (lane == 0) {
      nnz[t] = base;
      if (base > E) set_status(status, TWELL_ERR_CAPACITY);
    }
  }
}

struct REParams {
  const void *x, *Wu, *Wd;
  const uint16_t *idx;
  const void *val;
  const int32_t *nnz;
  void *y;
  int Tn, D, F, E, gated;
};

// One CTA (four warps) per token.  The row's entries are staged in shared
// memory; phase 1 (gated FFN): warp w computes u = x . W_up[n] for entries
// w, w + 4, ... (x in shared memory, warp shuffles only) and h = g u;
// phase 2: every thread accumulates y += h W_down[n] over its 16-byte slices
// of d_model, PB rows in flight.  fp32 accumulation, y rounded once.
template <class T, int VPL, int VPT>
__global__ void __launch_bounds__(RE_THREADS) rowell_updown_kernel(REParams p) {
  pdl_begin();
  constexpr int EV = Vec<T>::EV;
  __shared__ int s_n[RE_CHUNK];
  __shared__ float s_h[RE_CHUNK];
  __shared__ uint4 s_x[1024];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int NV = p.D / EV;
  const uint4 *x4 = (const uint4 *)p.x, *Wu4 = (const uint4 *)p.Wu, *Wd4 = (const uint4 *)p.Wd;
  if (p.gated)
    for (int v = tid; v < NV; v += blockDim.x) s_x[v] = x4[(size_t)t * NV + v];
  float2 acc[VPT][EV / 2];
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int e = 0; e < EV / 2; ++e) acc[v][e] = make_float2(0.f, 0.f);
  const int n_all = min(p.nnz[t], p.E);
  const uint16_t *ri = p.idx + (size_t)t * p.E;
  const T *rv = (const T *)p.val + (size_t)t * p.E;
  for (int c0 = 0; c0 < n_all; c0 += RE_CHUNK) {
    const int m = min(n_all - c0, RE_CHUNK);
    __syncthreads();  // the previous chunk is consumed (and s_x is written)
    for (int i = tid; i < m; i += blockDim.x) {  // (an index past F would be malformed: no-op)
      const int n = ri[c0 + i];
      s_n[i] = n < p.F ? n : 0;
      s_h[i] = n < p.F ? to_f(rv[c0 + i]) : 0.f;
    }
    __syncthreads();
    if (p.gated) {
      for (int i = w; i < m; i += RE_THREADS / 32) {
        uint4 r[VPL];
        warp_row<VPL>(Wu4 + (size_t)s_n[i] * NV, NV, true, r);
        const float u = warp_dot_smem<T, VPL>(s_x, NV, r);
        if (lane == 0) s_h[i] *= u;  // h = g u
      }
      __syncthreads();
    }
    for (int b0 = 0; b0 < m; b0 += PB) {
      const int nb = m - b0 < PB ? m - b0 : PB;
      uint4 r[PB][VPT];
      gather8<T, VPT, PB>(Wd4, s_n, b0, nb, NV, NV, r);
#pragma unroll
      for (int b = 0; b < PB; ++b) {
        if (b >= nb) break;
        const float h = s_h[b0 + b];
#pragma unroll
        for (int v = 0; v < VPT; ++v) axpy_vec<T>(acc[v], h, r[b][v]);
      }
    }
  }
  uint4 *yrow = (uint4 *)p.y + (size_t)t * NV;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int vi = tid + v * blockDim.x;
    if (vi < NV) stg_stream(yrow + vi, Vec<T>::pack(reinterpret_cast<const float *>(acc[v])));
  }
}

}  // namespace

cudaError_t launch_rowell_pack_dense(const void *H, int T, int F, int E, int dtype, uint16_t *idx,
                                     void *val, int32_t *nnz, int32_t *status, cudaStream_t s) {
  const int warps = 8;
  long blocks = ((long)T + warps - 1) / warps;
  if (blocks > 8L * num_sms()) blocks = 8L * num_sms();
  if (dtype == TWELL_BF16)
    launch_k(rowell_pack_dense_kernel<bf16>, (unsigned)blocks, warps * 32, 0, s, (const bf16 *)H,
             T, F, E, idx, (bf16 *)val, nnz, status);
  else
    launch_k(rowell_pack_dense_kernel<float>, (unsigned)blocks, warps * 32, 0, s,
             (const float *)H, T, F, E, idx, (float *)val, nnz, status);
  return cudaGetLastError();
}

cudaError_t launch_rowell_updown(const void *x, const void *Wu, const void *Wd, int T, int D,
                                 int F, int E, int dtype, const uint16_t *idx, const void *val,
                                 const int32_t *nnz, void *y, cudaStream_t s) {
  REParams p;
  p.x = x; p.Wu = Wu; p.Wd = Wd; p.idx = idx; p.val = val; p.nnz = nnz; p.y = y;
  p.Tn = T; p.D = D; p.F = F; p.E = E; p.gated = Wu != nullptr;
  const int EV = dtype == TWELL_BF16 ? 8 : 4;
  const int NV = D / EV;  // <= 1024 (checked by the caller)
  const int vpl = NV <= 32 ? 1 : NV <= 64 ? 2 : NV <= 128 ? 4 : NV <= 256 ? 8 : NV <= 512 ? 16 : 32;
  const int vpt = (NV + RE_THREADS - 1) / RE_THREADS;  // 1..8
#define RE_L(TT, L)                                                                            \
  do {                                                                                         \
    if (vpt <= 1) launch_k(rowell_updown_kernel<TT, L, 1>, T, RE_THREADS, 0, s, p);             \
    else if (vpt <= 2) launch_k(rowell_updown_kernel<TT, L, 2>, T, RE_THREADS, 0, s, p);        \
    else if (vpt <= 4) launch_k(rowell_updown_kernel<TT, L, 4>, T, RE_THREADS, 0, s, p);        \
    else launch_k(rowell_updown_kernel<TT, L, 8>, T, RE_THREADS, 0, s, p);                      \
  } while (0)
#define RE_T(TT)                                                                               \
  do {                                                                                         \
    switch (vpl) {                                                                             \
      case 1: RE_L(TT, 1); break;                                                              \
      case 2: RE_L(TT, 2); break;                                                              \
      case 4: RE_L(TT, 4); break;                                                              \
      case 8: RE_L(TT, 8); break;                                                              \
      case 16: RE_L(TT, 16); break;                                                            \
      default: RE_L(TT, 32); break;                                                            \
    }                                                                                          \
  } while (0)
  if (dtype == TWELL_BF16) RE_T(bf16);
  else RE_T(float);
#undef RE_T
#undef RE_L
  return cudaGetLastError();
}

}  // namespace twell

// updown.cu -- fused sparse up + down projection over TwELL.
//
// "Sparser, Faster, Lighter Transformer Language Models", technical summary
// section 2.B (inference): one fused kernel performs the up and down
// projections in a single pass from the gate activations stored in TwELL,
// keeping global-memory traffic low and working from registers and shared
// memory.
//
// Design (GB300): one CTA per token.  Thread i owns the 16-byte vectors
// i, i + blockDim, ... of the d_model axis, so every gathered weight row is read
// by the CTA as fully coalesced 128-bit loads.  x_t and the y_t accumulators
// stay in registers for the whole token.  The active pairs (neuron n, gate g)
// come from the token's TwELL slots, compacted into a shared-memory list.  Pairs
// are consumed in batches of 8: all 8 W_up and 8 W_down rows are requested
// before any is used (16 independent 128-bit loads per thread in flight), the 8
// partial dot products are reduced with a 9-shuffle transpose-reduction per
// warp plus one shared-memory pass across warps, then h = g * u and
// y += h * W_down[n].  Overflow rows and all-dense mode are left to the dense
// fallback.
#include "common.cuh"
#include "kernels.h"

namespace twell {

namespace {

constexpr int LIST_CAP = 2048;  // pairs staged per tile group
constexpr int PB = 8;           // pairs per batch

struct UDParams {
  const void *x, *Wu, *Wd;
  const uint8_t *idx, *nnz;
  const void *val;
  void *u_val, *y;
  int Tn, D, F, C, K, gated, train;
  const Ctl *ctl;
  int32_t *status;
};

template <class T> struct Vec;
template <> struct Vec<bf16> {
  static constexpr int EV = 8;
  static __device__ __forceinline__ void unpack(const uint4 &r, float *f) {
    f[0] = bf_lo(r.x); f[1] = bf_hi(r.x); f[2] = bf_lo(r.y); f[3] = bf_hi(r.y);
    f[4] = bf_lo(r.z); f[5] = bf_hi(r.z); f[6] = bf_lo(r.w); f[7] = bf_hi(r.w);
  }
  static __device__ __forceinline__ uint4 pack(const float *f) {
    return make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]),
                      pack_bf2(f[6], f[7]));
  }
};
template <> struct Vec<float> {
  static constexpr int EV = 4;
  static __device__ __forceinline__ void unpack(const uint4 &r, float *f) {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
  }
  static __device__ __forceinline__ uint4 pack(const float *f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// Dot product of the thread's slice of x with one gathered row (in registers).
template <class T, int VPT>
__device__ __forceinline__ float slice_dot(const float (&xr)[VPT][Vec<T>::EV],
                                           const uint4 (&w)[VPT]) {
  constexpr int EV = Vec<T>::EV;
  float s = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    float f[EV];
    Vec<T>::unpack(w[v], f);
#pragma unroll
    for (int e = 0; e < EV; ++e) s = fmaf(xr[v][e], f[e], s);
  }
  return s;
}

// Reduce 8 per-lane values across the warp; afterwards lane L holds the warp
// total of value (L >> 2) & 7.
__device__ __forceinline__ float warp_reduce8(float (&p)[PB]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 16;
    const float send = hi ? p[i] : p[i + 4];
    const float keep = hi ? p[i + 4] : p[i];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 8;
    const float send = hi ? p[i] : p[i + 2];
    const float keep = hi ? p[i + 2] : p[i];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  {
    const bool hi = lane & 4;
    const float send = hi ? p[0] : p[1];
    const float keep = hi ? p[1] : p[0];
    p[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  p[0] += __shfl_xor_sync(0xffffffffu, p[0], 2);
  p[0] += __shfl_xor_sync(0xffffffffu, p[0], 1);
  return p[0];
}

}  // namespace

template <class T, int VPT>
__global__ void __launch_bounds__(512) updown_fused_kernel(UDParams p) {
  constexpr int EV = Vec<T>::EV;
  __shared__ int s_n[LIST_CAP];
  __shared__ float s_g[LIST_CAP];
  __shared__ int s_slot[LIST_CAP];
  __shared__ int s_wsum[32];
  __shared__ float s_red[PB][33];
  __shared__ float s_u[PB];
  __shared__ int s_flag, s_total;

  if (p.ctl->dense) return;
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
  const int nt = p.F / p.C;
  const int NV = p.D / EV;

  // Overflow rows belong to the dense fallback.
  if (tid == 0) s_flag = 0;
  __syncthreads();
  for (int j = tid; j < nt; j += blockDim.x)
    if (p.nnz[(size_t)j * p.Tn + t] > p.K) s_flag = 1;
  __syncthreads();
  if (s_flag) return;

  const uint4 *xrow = (const uint4 *)p.x + (size_t)t * NV;
  float xr[VPT][EV], yr[VPT][EV];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int vi = tid + v * blockDim.x;
    uint4 r = make_uint4(0, 0, 0, 0);
    if (p.gated && vi < NV) r = xrow[vi];
    Vec<T>::unpack(r, xr[v]);
#pragma unroll
    for (int e = 0; e < EV; ++e) yr[v][e] = 0.f;
  }
  const uint4 *Wu4 = (const uint4 *)p.Wu, *Wd4 = (const uint4 *)p.Wd;
  const T *val = (const T *)p.val;

  int group = LIST_CAP / p.K;
  if (group > (int)blockDim.x) group = blockDim.x;
  for (int g0 = 0; g0 < nt; g0 += group) {
    // ---- compact this tile group's slots into the pair list -------------
    const int j = g0 + tid;
    const int cnt = (tid < group && j < nt) ? (int)p.nnz[(size_t)j * p.Tn + t] : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) s_wsum[w] = incl;
    __syncthreads();
    if (w == 0) {
      const int v = lane < nw ? s_wsum[lane] : 0;
      int wi = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += u;
      }
      if (lane < nw) s_wsum[lane] = wi - v;
      if (lane == 31) s_total = wi;
    }
    __syncthreads();
    const int off = s_wsum[w] + incl - cnt;
    const int P = s_total;
    if (cnt > 0) {
      const size_t s0 = ((size_t)j * p.Tn + t) * (size_t)p.K;
      for (int k = 0; k < cnt; ++k) {
        int c = p.idx[s0 + k];
        if (c >= p.C) {
          set_status(p.status, TWELL_ERR_INDEX);
          c = 0;
        }
        s_n[off + k] = j * p.C + c;
        s_g[off + k] = to_f(val[s0 + k]);
        s_slot[off + k] = (int)(s0 + k);
      }
    }
    __syncthreads();

    // ---- consume the pairs in batches of PB -------------------------------
    for (int b0 = 0; b0 < P; b0 += PB) {
      const int nb = P - b0 < PB ? P - b0 : PB;
      uint4 wd[PB][VPT];
      float h[PB];
      if (p.gated) {
        uint4 wu[PB][VPT];
#pragma unroll
        for (int b = 0; b < PB; ++b) {
          const size_t rb = (size_t)s_n[b0 + (b < nb ? b : 0)] * NV;
#pragma unroll
          for (int v = 0; v < VPT; ++v) {
            const int vi = tid + v * blockDim.x;
            const bool ok = b < nb && vi < NV;
            wu[b][v] = ok ? ldg_stream(Wu4 + rb + vi) : make_uint4(0, 0, 0, 0);
            wd[b][v] = ok ? ldg_stream(Wd4 + rb + vi) : make_uint4(0, 0, 0, 0);
          }
        }
        float pd[PB];
#pragma unroll
        for (int b = 0; b < PB; ++b) pd[b] = slice_dot<T, VPT>(xr, wu[b]);
        const float wsum = warp_reduce8(pd);
        if ((lane & 3) == 0) s_red[lane >> 2][w] = wsum;
        __syncthreads();
        if (tid < PB) {
          float u = 0.f;
          for (int q = 0; q < nw; ++q) u += s_red[tid][q];
          s_u[tid] = u;
          if (p.train && tid < nb) ((T *)p.u_val)[s_slot[b0 + tid]] = from_f<T>(u);
        }
        __syncthreads();
#pragma unroll
        for (int b = 0; b < PB; ++b) h[b] = b < nb ? s_g[b0 + b] * s_u[b] : 0.f;
      } else {
#pragma unroll
        for (int b = 0; b < PB; ++b) {
          const size_t rb = (size_t)s_n[b0 + (b < nb ? b : 0)] * NV;
#pragma unroll
          for (int v = 0; v < VPT; ++v) {
            const int vi = tid + v * blockDim.x;
            wd[b][v] = (b < nb && vi < NV) ? ldg_stream(Wd4 + rb + vi) : make_uint4(0, 0, 0, 0);
          }
          h[b] = b < nb ? s_g[b0 + b] : 0.f;
        }
      }
#pragma unroll
      for (int b = 0; b < PB; ++b) {
        if (b >= nb) break;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          float f[EV];
          Vec<T>::unpack(wd[b][v], f);
#pragma unroll
          for (int e = 0; e < EV; ++e) yr[v][e] = fmaf(h[b], f[e], yr[v][e]);
        }
      }
    }
    __syncthreads();  // the list is rewritten by the next group
  }

  uint4 *yrow = (uint4 *)p.y + (size_t)t * NV;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int vi = tid + v * blockDim.x;
    if (vi < NV) yrow[vi] = Vec<T>::pack(yr[v]);
  }
}

cudaError_t launch_updown_fused(const FwdArgs &a, cudaStream_t s) {
  UDParams p;
  p.x = a.x; p.Wu = a.Wu; p.Wd = a.Wd; p.idx = a.tw.idx; p.nnz = a.tw.nnz; p.val = a.tw.val;
  p.u_val = a.tw.u_val; p.y = a.y; p.Tn = a.T; p.D = a.D; p.F = a.F; p.C = a.C; p.K = a.K;
  p.gated = a.gated; p.train = a.train && a.gated; p.ctl = a.ws.ctl; p.status = a.tw.status;
  const int EV = a.dtype == TWELL_BF16 ? 8 : 4;
  const int NV = a.D / EV;
  const int vpt = NV <= 512 ? 1 : 2;  // at most 512 threads, NV <= 1024 checked by the caller
  int threads = (NV + vpt - 1) / vpt;
  threads = (threads + 31) / 32 * 32;
  if (a.dtype == TWELL_BF16) {
    if (vpt == 1) updown_fused_kernel<bf16, 1><<<a.T, threads, 0, s>>>(p);
    else updown_fused_kernel<bf16, 2><<<a.T, threads, 0, s>>>(p);
  } else {
    if (vpt == 1) updown_fused_kernel<float, 1><<<a.T, threads, 0, s>>>(p);
    else updown_fused_kernel<float, 2><<<a.T, threads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace twell

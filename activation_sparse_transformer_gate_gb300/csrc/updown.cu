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
// before any is used, the 8 partial dot products are reduced with a 9-shuffle
// transpose-reduction per warp plus one shared-memory pass across warps, then
// h = g * u and y += h * W_down[n].  The next batch's W_up rows are requested
// before the reduction and its W_down rows right after the accumulation, so
// loads stay in flight across the barriers.  All-dense mode (and overflow rows
// when there are many) is left to the tensor-core dense-row GEMMs; a few
// overflow rows are handled here from the wide-tile buffer.
#include "common.cuh"
#include "gather.cuh"
#include "kernels.h"

namespace twell {

namespace {

struct UDParams {
  const void *x, *Wu, *Wd;
  const uint8_t *idx, *nnz;
  const void *val, *wide;
  void *u_val, *y, *g_fb, *u_fb;
  const int32_t *pos;
  int Tn, D, F, C, K, gated, train, cap;
  const Ctl *ctl;
  int32_t *status;
};

}  // namespace

// One CTA per token.  Rows that run on the dense GEMM path (all-dense mode, or
// overflow rows when there are many) are skipped; an overflow row handled
// here takes its overflowing tiles from the wide-tile buffer and also writes
// its dense backup row (g_fb, and u_fb when training).
template <class T, int VPT>
__global__ void __launch_bounds__(512) updown_fused_kernel(UDParams p) {
  constexpr int EV = Vec<T>::EV;
  __shared__ int s_n[LIST_CAP];
  __shared__ float s_g[LIST_CAP];
  __shared__ int s_slot[LIST_CAP];
  __shared__ int s_wsum[32];
  __shared__ float s_red[PB][33];
  __shared__ float s_tot[PB];
  __shared__ int s_total;

  if (p.ctl->dense) return;
  const int t = blockIdx.x;
  const int ps = p.pos[t];
  const bool ovf = ps >= 0;
  if (ovf && p.ctl->ovf_gemm) return;
  const int tid = threadIdx.x;
  const int nt = p.F / p.C;
  const int NV = p.D / EV;
  const bool fb = ovf && ps < p.cap;
  if (fb) {  // dense backup row(s): zeros, the active values are scattered below
    const int rv = p.F * (int)sizeof(T) / 16;
    uint4 *g4 = (uint4 *)((T *)p.g_fb + (size_t)ps * p.F);
    uint4 *u4 = p.train ? (uint4 *)((T *)p.u_fb + (size_t)ps * p.F) : nullptr;
    for (int v = tid; v < rv; v += blockDim.x) {
      g4[v] = make_uint4(0, 0, 0, 0);
      if (u4) u4[v] = make_uint4(0, 0, 0, 0);
    }
  }

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
  PairSource<T> src;
  src.idx = p.idx; src.nnz = p.nnz; src.val = (const T *)p.val; src.Tn = p.Tn; src.C = p.C;
  src.K = p.K; src.t = t;
  src.dense = ovf ? (const T *)p.wide + (size_t)t * p.C : nullptr;
  src.dense_tile = (size_t)p.Tn * p.C;
  src.dense_all = false;
  src.neg_slots = ovf;

  int group = LIST_CAP / (ovf ? p.C : p.K);
  if (group > (int)blockDim.x) group = blockDim.x;
  for (int g0 = 0; g0 < nt; g0 += group) {
    const int P = build_pairs(src, g0, group, nt, s_n, s_g, s_slot, s_wsum, &s_total, p.status);
    if (fb)
      for (int i = tid; i < P; i += blockDim.x)
        if (s_slot[i] != PAD_SLOT) ((T *)p.g_fb)[(size_t)ps * p.F + s_n[i]] = from_f<T>(s_g[i]);
    if (P > 0) {
      uint4 wu[PB][VPT], wd[PB][VPT];
      int nb = P < PB ? P : PB;
      if (p.gated) gather8<T, VPT>(Wu4, s_n, 0, nb, NV, wu);
      gather8<T, VPT>(Wd4, s_n, 0, nb, NV, wd);
      for (int b0 = 0; b0 < P; b0 += PB) {
        const int b1 = b0 + PB;
        const int nb_next = P - b1 < PB ? P - b1 : PB;
        float h[PB];
        if (p.gated) {
          float pd[PB];
#pragma unroll
          for (int b = 0; b < PB; ++b) pd[b] = slice_dot<T, VPT>(xr, wu[b]);
          // the next batch's W_up rows are in flight during the reduction
          if (nb_next > 0) gather8<T, VPT>(Wu4, s_n, b1, nb_next, NV, wu);
          float u[PB];
          block_reduce8(pd, u, s_red, s_tot);
#pragma unroll
          for (int b = 0; b < PB; ++b) h[b] = b < nb ? s_g[b0 + b] * u[b] : 0.f;
          if (p.train && tid < nb) {
            const int sl = s_slot[b0 + tid];
            float uv = 0.f;
#pragma unroll
            for (int b = 0; b < PB; ++b)
              if (b == tid) uv = u[b];
            if (sl >= 0) ((T *)p.u_val)[sl] = from_f<T>(uv);
            else if (fb && sl != PAD_SLOT) ((T *)p.u_fb)[(size_t)ps * p.F + (-1 - sl)] = from_f<T>(uv);
          }
        } else {
#pragma unroll
          for (int b = 0; b < PB; ++b) h[b] = b < nb ? s_g[b0 + b] : 0.f;
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
        if (nb_next > 0) gather8<T, VPT>(Wd4, s_n, b1, nb_next, NV, wd);
        nb = nb_next;
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
  p.wide = a.ws.wide; p.u_val = a.tw.u_val; p.y = a.y; p.g_fb = a.tw.g_fb; p.u_fb = a.tw.u_fb;
  p.pos = a.ws.pos; p.Tn = a.T; p.D = a.D; p.F = a.F; p.C = a.C; p.K = a.K; p.gated = a.gated;
  p.train = a.train && a.gated; p.cap = a.tw.ovf_cap; p.ctl = a.ws.ctl; p.status = a.tw.status;
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

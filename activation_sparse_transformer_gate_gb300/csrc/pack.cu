// pack.cu -- TwELL packing of a dense activation matrix, the overflow-row
// compaction that turns TwELL into the hybrid format, and row gathers.
//
// "Sparser, Faster, Lighter Transformer Language Models", technical summary
// section 2.A: TwELL keeps K (index, value) slots per (row, tile of C
// columns); section 2.A hybrid format: rows that overflow their slots go to a
// dense backup matrix; section 2.B: conversion from TwELL to the hybrid form.
#include "common.cuh"
#include "kernels.h"

namespace twell {

// One warp packs one (row, tile).  Lane l holds columns l + 32e (e < E), so the
// warp reads 32 consecutive elements per step; the slot of an active column
// is its rank among the active columns, counted with ballot + popc.
template <class T, int E>
__global__ void pack_dense_kernel(const T *__restrict__ H, int Tn, int F, int K,
                                  uint8_t *__restrict__ idx, T *__restrict__ val,
                                  uint8_t *__restrict__ nnz) {
  const int lane = threadIdx.x & 31;
  const long warp = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int C = 32 * E;
  const int nt = F / C;
  if (warp >= (long)Tn * nt) return;
  const int t = (int)(warp % Tn), j = (int)(warp / Tn);
  const T *row = H + (size_t)t * F + (size_t)j * C;
  T raw[E];
  unsigned m[E];
  int cnt = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    raw[e] = row[lane + 32 * e];
    m[e] = __ballot_sync(0xffffffffu, to_f(raw[e]) > 0.f);
    cnt += __popc(m[e]);
  }
  const size_t s0 = ((size_t)j * Tn + t) * (size_t)K;
  const unsigned lt = (1u << lane) - 1u;
  int before = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if ((m[e] >> lane) & 1u) {
      int r = before + __popc(m[e] & lt);
      if (r < K) {
        idx[s0 + r] = (uint8_t)(lane + 32 * e);
        val[s0 + r] = raw[e];
      }
    }
    before += __popc(m[e]);
  }
  const int filled = cnt < K ? cnt : K;
  for (int k = lane; k < K; k += 32)
    if (k >= filled) {
      idx[s0 + k] = 0xFF;
      val[s0 + k] = from_f<T>(0.f);
    }
  if (lane == 0) nnz[(size_t)j * Tn + t] = (uint8_t)cnt;
}

cudaError_t launch_pack_dense(const void *H, const twell_t &tw, cudaStream_t s) {
  const long warps = (long)tw.T * (tw.F / tw.C);
  const int threads = 256;
  const long blocks = (warps * 32 + threads - 1) / threads;
  const int E = tw.C / 32;
#define TW_PD(TT, EE)                                                                          \
  pack_dense_kernel<TT, EE><<<(unsigned)blocks, threads, 0, s>>>(                             \
      (const TT *)H, tw.T, tw.F, tw.K, tw.idx, (TT *)tw.val, tw.nnz)
  if (tw.dtype == TWELL_BF16) {
    if (E == 1) TW_PD(bf16, 1); else if (E == 2) TW_PD(bf16, 2); else TW_PD(bf16, 4);
  } else {
    if (E == 1) TW_PD(float, 1); else if (E == 2) TW_PD(float, 2); else TW_PD(float, 4);
  }
#undef TW_PD
  return cudaGetLastError();
}

// Hybrid split (one CTA of 1024 threads): a row overflows iff one of its tiles
// has nnz > K.  Rows are visited in ascending order, 1024 at a time; a
// ballot/popc block scan gives each overflow row its list position, so the
// list is ascending and deterministic.  Writes the caller's list (first
// ovf_cap entries) and count, and -- when a workspace is given -- the full
// dense-path row list, each row's position, and the control block that picks
// hybrid or all-dense mode.
__global__ void __launch_bounds__(1024)
overflow_compact_kernel(const uint8_t *__restrict__ nnz, int Tn, int nt, int K, int cap,
                        int32_t *__restrict__ ovf_rows, int32_t *__restrict__ n_ovf,
                        int32_t *status, Ctl *ctl, int32_t *__restrict__ rows,
                        int32_t *__restrict__ pos, float dense_switch) {
  __shared__ int warp_cnt[32];
  __shared__ int warp_off[32];
  __shared__ int total;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int running = 0;
  for (int base = 0; base < Tn; base += blockDim.x) {
    const int t = base + tid;
    int flag = 0;
    if (t < Tn)
      for (int j = 0; j < nt; ++j)
        if (nnz[(size_t)j * Tn + t] > K) {
          flag = 1;
          break;
        }
    const unsigned b = __ballot_sync(0xffffffffu, flag);
    if (lane == 0) warp_cnt[w] = __popc(b);
    __syncthreads();
    if (w == 0) {
      const int nw = blockDim.x >> 5;
      int v = lane < nw ? warp_cnt[lane] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      warp_off[lane] = incl - v;
      if (lane == 31) total = incl;
    }
    __syncthreads();
    const int p = running + warp_off[w] + __popc(b & ((1u << lane) - 1u));
    if (t < Tn) {
      if (flag) {
        if (rows) rows[p] = t;
        if (p < cap) ovf_rows[p] = t;
      }
      if (pos) pos[t] = flag ? p : -1;
    }
    running += total;
    __syncthreads();
  }
  if (tid == 0) {
    *n_ovf = running;
    if (running > cap) set_status(status, TWELL_ERR_CAPACITY);
    if (ctl) {
      const int dense = (float)running > dense_switch * (float)Tn ? 1 : 0;
      ctl->n_ovf = running;
      ctl->dense = dense;
      ctl->n_rows = dense ? Tn : running;
    }
  }
}

cudaError_t launch_overflow_compact(const twell_t &tw, const Workspace *ws, float dense_switch,
                                    cudaStream_t s) {
  overflow_compact_kernel<<<1, 1024, 0, s>>>(
      tw.nnz, tw.T, tw.F / tw.C, tw.K, tw.ovf_cap, tw.ovf_rows, tw.n_ovf, tw.status,
      ws ? ws->ctl : nullptr, ws ? ws->rows : nullptr, ws ? ws->pos : nullptr, dense_switch);
  return cudaGetLastError();
}

// g_fb[i] = H[ovf_rows[i]] for i < min(n_ovf, ovf_cap); 16-byte copies.
__global__ void copy_fb_rows_kernel(const uint4 *__restrict__ H, int row_vecs, int cap,
                                    const int32_t *__restrict__ ovf_rows,
                                    const int32_t *__restrict__ n_ovf, uint4 *__restrict__ g_fb) {
  const int n = min(*n_ovf, cap);
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const uint4 *src = H + (size_t)ovf_rows[i] * row_vecs;
    uint4 *dst = g_fb + (size_t)i * row_vecs;
    for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) dst[v] = src[v];
  }
}

cudaError_t launch_copy_fb_rows(const void *H, const twell_t &tw, cudaStream_t s) {
  if (tw.ovf_cap <= 0) return cudaSuccess;
  const int es = tw.dtype == TWELL_BF16 ? 2 : 4;
  const int row_vecs = tw.F * es / 16;
  int blocks = tw.ovf_cap < tw.T ? tw.ovf_cap : tw.T;
  if (blocks > 1024) blocks = 1024;
  copy_fb_rows_kernel<<<blocks, 256, 0, s>>>((const uint4 *)H, row_vecs, tw.ovf_cap,
                                             tw.ovf_rows, tw.n_ovf, (uint4 *)tw.g_fb);
  return cudaGetLastError();
}

// dst[m] = src[rows[m]] for the dense-path rows (hybrid mode only; in all-dense
// mode the consumers read src directly).
__global__ void gather_rows_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                   int row_vecs, const Ctl *__restrict__ ctl,
                                   const int32_t *__restrict__ rows) {
  if (ctl->dense) return;
  const int n = ctl->n_rows;
  for (int m = blockIdx.x; m < n; m += gridDim.x) {
    const uint4 *a = src + (size_t)rows[m] * row_vecs;
    uint4 *b = dst + (size_t)m * row_vecs;
    for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) b[v] = a[v];
  }
}

cudaError_t launch_gather_rows(const void *src, void *dst, const Workspace &ws, int T, int D,
                               int dtype, cudaStream_t s) {
  const int es = dtype == TWELL_BF16 ? 2 : 4;
  int blocks = T < 1216 ? T : 1216;
  gather_rows_kernel<<<blocks, 256, 0, s>>>((const uint4 *)src, (uint4 *)dst, D * es / 16, ws.ctl,
                                            ws.rows);
  return cudaGetLastError();
}

}  // namespace twell

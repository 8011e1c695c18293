// pack.cu -- TwELL packing of a dense activation matrix, the overflow-row
// compaction that turns TwELL into the hybrid format, and the small row
// kernels around it.
//
// "Sparser, Faster, Lighter Transformer Language Models", technical summary
// section 2.A: TwELL keeps K (index, value) slots per (row, tile of C
// columns); section 2.A hybrid format: rows that overflow their slots go to a
// dense backup matrix; section 2.B: conversion from TwELL to the hybrid form.
#include <cuda_fp16.h>

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
  pdl_begin();
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
  launch_k(pack_dense_kernel<TT, EE>, (unsigned)blocks, threads, 0, s, (const TT *)H, tw.T,    \
           tw.F, tw.K, tw.idx, (TT *)tw.val, tw.nnz)
  if (tw.dtype == TWELL_BF16) {
    if (E == 1) TW_PD(bf16, 1); else if (E == 2) TW_PD(bf16, 2); else TW_PD(bf16, 4);
  } else {
    if (E == 1) TW_PD(float, 1); else if (E == 2) TW_PD(float, 2); else TW_PD(float, 4);
  }
#undef TW_PD
  return cudaGetLastError();
}

// Mode decisions taken on the device after the overflow rows are counted.
// All-dense when too many rows overflow, or when the slots the gate epilogue
// wrote (active entries, at most K per row and tile, so overflow rows count
// little) exceed dense_density * T * F: gathers then cost more than GEMMs.
// Backward (dh_density > 0): dh of the rows left to the gathers comes from
// one dense GEMM read at the slots when the slots exceed dh_density * T * F
// (each active entry costs the SDDMM a d_model row; the GEMM costs the same
// per entry of the whole T x F product).
// The dense path takes at most rows_cap rows (the workspace's dense-row
// buffers): no all-dense mode when rows_cap < Tn, and overflow rows beyond it
// stay on the gathers.
__device__ __forceinline__ void write_ctl(Ctl *ctl, int n_ovf, int Tn, int F, float dense_switch,
                                          float dense_density, float dh_density, int rows_cap) {
  const double TF = (double)Tn * (double)F;
  const bool too_dense = dense_density > 0.f && (double)ctl->slots > (double)dense_density * TF;
  const int dense =
      (((float)n_ovf > dense_switch * (float)Tn || too_dense) && Tn <= rows_cap) ? 1 : 0;
  const int og = (!dense && n_ovf >= OVF_GEMM_MIN && n_ovf <= rows_cap) ? 1 : 0;
  ctl->n_ovf = n_ovf;
  ctl->dense = dense;
  ctl->ovf_gemm = og;
  ctl->n_rows = dense ? Tn : (og ? n_ovf : 0);
  ctl->dh_gemm = (!dense && dh_density > 0.f && (double)ctl->slots > (double)dh_density * TF) ? 1 : 0;
}

// Hybrid split from nnz (one CTA of 1024 threads, no workspace): a row
// overflows iff one of its tiles has nnz > K.  Rows are visited in ascending
// order, 1024 at a time; a ballot/popc block scan gives each overflow row its
// list position, so the list is ascending and deterministic.
__global__ void __launch_bounds__(1024)
overflow_compact_kernel(const uint8_t *__restrict__ nnz, int Tn, int nt, int K, int cap,
                        int32_t *__restrict__ ovf_rows, int32_t *__restrict__ n_ovf,
                        int32_t *status) {
  pdl_begin();
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
    if (t < Tn && flag && p < cap) ovf_rows[p] = t;
    running += total;
    __syncthreads();
  }
  if (tid == 0) {
    *n_ovf = running;
    if (running > cap) set_status(status, TWELL_ERR_CAPACITY);
  }
}

// Hybrid split from the overflow-row bitmap (one CTA of 1024 threads).  Each
// thread owns one 32-row word per round; a block scan of the word popcounts
// gives each overflow row its ascending list position.
__global__ void __launch_bounds__(1024)
overflow_scan_kernel(const uint32_t *__restrict__ bits, int Tn, int cap,
                     int32_t *__restrict__ ovf_rows, int32_t *__restrict__ n_ovf, int32_t *status,
                     Ctl *ctl, int32_t *__restrict__ rows, int32_t *__restrict__ pos,
                     int F, float dense_switch, float dense_density,
                     const unsigned long long *__restrict__ slot_parts, int n_parts,
                     float dh_density, int rows_cap) {
  pdl_begin();
  __shared__ int warp_off[32];
  __shared__ int word_off[1024];
  __shared__ int total;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int words = (Tn + 31) / 32;
  int running = 0;
  for (int base = 0; base < words; base += 1024) {
    const int wi = base + tid;
    const uint32_t word = wi < words ? bits[wi] : 0u;
    const int c = __popc(word);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_off[w] = incl;
    __syncthreads();
    if (w == 0) {
      const int v = warp_off[lane];
      int wi2 = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, wi2, o);
        if (lane >= o) wi2 += u;
      }
      warp_off[lane] = wi2 - v;
      if (lane == 31) total = wi2;
    }
    __syncthreads();
    const int off = running + warp_off[w] + incl - c;
    word_off[tid] = off;
    uint32_t m = word;
    int k = 0;
    while (m) {  // list entries in ascending row order
      const int b = __ffs(m) - 1;
      m &= m - 1;
      const int t = wi * 32 + b;
      rows[off + k] = t;
      if (ovf_rows && off + k < cap) ovf_rows[off + k] = t;
      ++k;
    }
    __syncthreads();
    const int r0 = base * 32;  // positions of every row (coalesced)
    for (int r = tid; r < 1024 * 32; r += 1024) {
      const int t = r0 + r;
      if (t >= Tn) break;
      const uint32_t wd = bits[t >> 5];
      const int b = t & 31;
      pos[t] = ((wd >> b) & 1u) ? word_off[r >> 5] + __popc(wd & ((1u << b) - 1u)) : -1;
    }
    running += total;
    __syncthreads();
  }
  if (tid == 0) {
    if (slot_parts) {  // slot count from per-block partial sums (else the gate epilogue's)
      unsigned long long sl = 0;
      for (int i = 0; i < n_parts; ++i) sl += slot_parts[i];
      ctl->slots = sl;
    }
    if (n_ovf) *n_ovf = running;
    if (running > cap) set_status(status, TWELL_ERR_CAPACITY);
    write_ctl(ctl, running, Tn, F, dense_switch, dense_density, dh_density, rows_cap);
  }
}

cudaError_t launch_overflow_compact(const twell_t &tw, const Workspace *ws, float dense_switch,
                                    cudaStream_t s, bool write_user, float dense_density,
                                    const unsigned long long *slot_parts, int n_parts,
                                    float dh_density) {
  if (ws) {
    launch_k(overflow_scan_kernel, 1, 1024, 0, s, ws->ovf_bits, tw.T, tw.ovf_cap,
             write_user ? tw.ovf_rows : nullptr, write_user ? tw.n_ovf : nullptr, tw.status,
             ws->ctl, ws->rows, ws->pos, tw.F, dense_switch, dense_density, slot_parts, n_parts,
             dh_density, ws->dense_bufs ? ws->rp : 0);
    return cudaGetLastError();
  }
  launch_k(overflow_compact_kernel, 1, 1024, 0, s, tw.nnz, tw.T, tw.F / tw.C, tw.K, tw.ovf_cap,
           tw.ovf_rows, tw.n_ovf, tw.status);
  return cudaGetLastError();
}

// Overflow-row bitmap from nnz: a block per 32-row bitmap word at a time,
// warp g taking tiles g, g + 8, ... of the word's rows (one row per lane,
// reads coalesced across the warp); the warps' ballots are OR-ed and the word
// written whole (no zeroing, no atomics).  With slot_parts: each block's
// number of slots in use, sum of min(nnz, K) as the gate epilogue counts it.
__global__ void __launch_bounds__(256)
    flags_from_nnz_kernel(const uint8_t *__restrict__ nnz, int Tn, int nt, int K,
                          uint32_t *__restrict__ bits,
                          unsigned long long *__restrict__ slot_parts,
                          int32_t *__restrict__ zero, long zero_n) {
  pdl_begin();
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < zero_n;
       i += (long)gridDim.x * blockDim.x)
    zero[i] = 0;
  __shared__ uint32_t s_mask[8];
  __shared__ unsigned long long s_part[8];
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int words = (Tn + 31) / 32;
  unsigned long long mine = 0;
  for (int wd = blockIdx.x; wd < words; wd += gridDim.x) {  // uniform per block
    const int t = wd * 32 + lane;
    bool over = false;
    if (t < Tn) {
      for (int j = g; j < nt; j += 8) {
        const int c = nnz[(size_t)j * Tn + t];
        over |= c > K;
        mine += (unsigned long long)(c < K ? c : K);
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, over);
    if (lane == 0) s_mask[g] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t wm = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) wm |= s_mask[i];
      bits[wd] = wm;
    }
    __syncthreads();  // s_mask is rewritten for the next word
  }
  if (!slot_parts) return;  // uniform
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mine += __shfl_down_sync(0xffffffffu, mine, o);
  if (lane == 0) s_part[g] = mine;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long b = 0;
    for (int i = 0; i < 8; ++i) b += s_part[i];
    slot_parts[blockIdx.x] = b;
  }
}

int flags_blocks(int T) {
  const int words = (T + 31) / 32;
  const int cap = 4 * num_sms() < SLOT_PARTS_MAX ? 4 * num_sms() : SLOT_PARTS_MAX;
  return words < cap ? words : cap;
}

cudaError_t launch_flags_from_nnz(const twell_t &tw, uint32_t *bits,
                                  unsigned long long *slot_parts, cudaStream_t s, int32_t *zero,
                                  long zero_n) {
  launch_k(flags_from_nnz_kernel, flags_blocks(tw.T), 256, 0, s, tw.nnz, tw.T, tw.F / tw.C, tw.K,
           bits, slot_parts, zero, zero ? zero_n : 0L);
  return cudaGetLastError();
}

// g_fb[i] = H[ovf_rows[i]] for i < min(n_ovf, ovf_cap); 16-byte copies.
__global__ void copy_fb_rows_kernel(const uint4 *__restrict__ H, int row_vecs, int cap,
                                    const int32_t *__restrict__ ovf_rows,
                                    const int32_t *__restrict__ n_ovf, uint4 *__restrict__ g_fb) {
  pdl_begin();
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
  launch_k(copy_fb_rows_kernel, blocks, 256, 0, s, (const uint4 *)H, row_vecs, tw.ovf_cap,
           tw.ovf_rows, tw.n_ovf, (uint4 *)tw.g_fb);
  return cudaGetLastError();
}

// dst[m] = src[rows[m]] for the overflow rows when they take the dense GEMM
// path (in all-dense mode the GEMMs read src directly), then zero rows up to
// the next multiple of 128: a GEMM that contracts over these rows reads them.
__global__ void gather_rows_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                   int row_vecs, const Ctl *__restrict__ ctl,
                                   const int32_t *__restrict__ rows) {
  pdl_begin();
  if (ctl->dense || !ctl->ovf_gemm) return;
  const int n = ctl->n_rows;
  const int npad = (n + 127) / 128 * 128;
  for (int m = blockIdx.x; m < npad; m += gridDim.x) {
    uint4 *b = dst + (size_t)m * row_vecs;
    if (m < n) {
      const uint4 *a = src + (size_t)rows[m] * row_vecs;
      for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) b[v] = a[v];
    } else {
      for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) b[v] = make_uint4(0, 0, 0, 0);
    }
  }
}

cudaError_t launch_gather_rows(const void *src, void *dst, const Workspace &ws, int T, int D,
                               int dtype, cudaStream_t s) {
  const int es = dtype == TWELL_BF16 ? 2 : 4;
  // Usually idle (no overflow-row GEMM): a small grid that loops over the rows.
  int blocks = T < 2 * num_sms() ? T : 2 * num_sms();
  launch_k(gather_rows_kernel, blocks, 256, 0, s, (const uint4 *)src, (uint4 *)dst, D * es / 16,
           ws.ctl, ws.rows);
  return cudaGetLastError();
}

// Dense backup rows of the overflow rows (when they do not take the dense GEMM
// path): zeros, then the slots of the tiles that fit and the wide tiles of
// those that overflow.  One CTA per overflow-list position.
template <class T>
__global__ void assemble_fb_rows_kernel(const Ctl *__restrict__ ctl,
                                        const int32_t *__restrict__ rows,
                                        const uint8_t *__restrict__ idx,
                                        const uint8_t *__restrict__ nnz, const T *__restrict__ val,
                                        const T *__restrict__ wide, T *__restrict__ g_fb, int Tn,
                                        int F, int C, int K, int cap) {
  pdl_begin();
  if (ctl->dense || ctl->ovf_gemm) return;
  const int n_fb = min(ctl->n_ovf, cap);
  for (int i = blockIdx.x; i < n_fb; i += gridDim.x) {
    const int t = rows[i];
    T *row = g_fb + (size_t)i * F;
    for (int n = threadIdx.x; n < F; n += blockDim.x) row[n] = from_f<T>(0.f);
    __syncthreads();
    for (int j = threadIdx.x; j < F / C; j += blockDim.x) {
      const size_t tj = (size_t)j * Tn + t;
      const int cnt = nnz[tj];
      if (cnt > K) {
        for (int c = 0; c < C; ++c) row[(size_t)j * C + c] = wide[tj * C + c];
      } else {
        for (int k = 0; k < cnt; ++k) {
          const int c = idx[tj * K + k];
          if (c < C) row[(size_t)j * C + c] = val[tj * K + k];
        }
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_assemble_fb_rows(const FwdArgs &a, cudaStream_t s) {
  if (a.tw.ovf_cap <= 0) return cudaSuccess;
  int blocks = a.tw.ovf_cap < a.T ? a.tw.ovf_cap : a.T;
  if (blocks > OVF_GEMM_MIN) blocks = OVF_GEMM_MIN;
  if (a.dtype == TWELL_BF16)
    launch_k(assemble_fb_rows_kernel<bf16>, blocks, 256, 0, s,
        a.ws.ctl, a.ws.rows, a.tw.idx, a.tw.nnz, (const bf16 *)a.tw.val, (const bf16 *)a.ws.wide,
        (bf16 *)a.tw.g_fb, a.T, a.F, a.C, a.K, a.tw.ovf_cap);
  else
    launch_k(assemble_fb_rows_kernel<float>, blocks, 256, 0, s,
        a.ws.ctl, a.ws.rows, a.tw.idx, a.tw.nnz, (const float *)a.tw.val,
        (const float *)a.ws.wide, (float *)a.tw.g_fb, a.T, a.F, a.C, a.K, a.tw.ovf_cap);
  return cudaGetLastError();
}

// All-dense training forward: u at the slots of the non-overflow rows, read
// from the u rows the dense gate+up GEMM wrote.  One thread per (tile, row).
template <class T>
__global__ void fill_u_slots_kernel(const Ctl *__restrict__ ctl, const int32_t *__restrict__ pos,
                                    const uint8_t *__restrict__ idx,
                                    const uint8_t *__restrict__ nnz, const T *__restrict__ urows,
                                    T *__restrict__ u_val, int Tn, int F, int C, int K) {
  pdl_begin();
  if (!ctl->dense) return;
  const long total = (long)Tn * (F / C);
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int t = (int)(i % Tn), j = (int)(i / Tn);
    if (pos[t] >= 0) continue;  // overflow rows keep u in the dense backup
    const int n = nnz[i] < K ? nnz[i] : K;
    for (int k = 0; k < n; ++k) {
      const int c = idx[i * K + k];
      if (c < C) u_val[i * K + k] = urows[(size_t)t * F + (size_t)j * C + c];
    }
  }
}

cudaError_t launch_fill_u_slots(const FwdArgs &a, cudaStream_t s) {
  const long total = (long)a.T * (a.F / a.C);
  long blocks = (total + 255) / 256;  // usually idle (all-dense mode only)
  if (blocks > 4L * num_sms()) blocks = 4L * num_sms();
  if (a.dtype == TWELL_BF16)
    launch_k(fill_u_slots_kernel<bf16>, (unsigned)blocks, 256, 0, s,
        a.ws.ctl, a.ws.pos, a.tw.idx, a.tw.nnz, (const bf16 *)a.ws.urows, (bf16 *)a.tw.u_val,
        a.T, a.F, a.C, a.K);
  else
    launch_k(fill_u_slots_kernel<float>, (unsigned)blocks, 256, 0, s,
        a.ws.ctl, a.ws.pos, a.tw.idx, a.tw.nnz, (const float *)a.ws.urows, (float *)a.tw.u_val,
        a.T, a.F, a.C, a.K);
  return cudaGetLastError();
}

// Eight bf16 values (one 16-byte vector) as fp16; sets *big when one of them
// lies beyond the fp16 range (the conversion is exact inside it, down to
// 2^-14, and keeps fp16's subnormal spacing below).
__device__ __forceinline__ uint4 bf16x8_to_f16(const uint4 &v, bool &big) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = bf_lo(w[i]), b = bf_hi(w[i]);
    big |= fabsf(a) > 65504.f || fabsf(b) > 65504.f;
    __half2 h = __floats2half2_rn(a, b);
    o[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Backward, dense-path rows (all rows in all-dense mode, else the overflow
// rows when they take the GEMMs): copy the rows' dy and x as fp16 (the operands of the fp16 tensor-core GEMMs; in
// all-dense mode row m is token m), zero rows up to the next multiple of 128.
// One launch, idle when there are no such rows.
__global__ void bwd_prep_rows_kernel(const Ctl *__restrict__ ctl, const int32_t *__restrict__ rows,
                                     const uint4 *__restrict__ dy, const uint4 *__restrict__ x,
                                     uint4 *__restrict__ dyg, uint4 *__restrict__ xg,
                                     int row_vecs, int32_t *status) {
  pdl_begin();
  const int n = ctl->n_rows;
  if (n == 0) return;
  const bool dense = ctl->dense != 0;
  const int npad = (n + 127) / 128 * 128;
  bool big = false;
  for (int m = blockIdx.x; m < npad; m += gridDim.x) {
    uint4 *a = dyg + (size_t)m * row_vecs, *b = xg + (size_t)m * row_vecs;
    if (m < n) {
      const int t = dense ? m : rows[m];
      const uint4 *sa = dy + (size_t)t * row_vecs, *sb = x + (size_t)t * row_vecs;
      for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
        a[v] = bf16x8_to_f16(sa[v], big);
        b[v] = bf16x8_to_f16(sb[v], big);
      }
    } else {
      for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) a[v] = b[v] = make_uint4(0, 0, 0, 0);
    }
  }
  if (big) set_status(status, TWELL_ERR_RANGE);
}

// fp16 copies of up to three bf16 matrices of `vecs` 16-byte vectors each,
// when the dense path has rows (else every CTA returns at once).
__global__ void to_f16_kernel(const uint4 *__restrict__ s0, uint4 *__restrict__ d0,
                              const uint4 *__restrict__ s1, uint4 *__restrict__ d1,
                              const uint4 *__restrict__ s2, uint4 *__restrict__ d2, size_t vecs,
                              const Ctl *__restrict__ ctl, int32_t *status) {
  pdl_begin();
  if (ctl->n_rows == 0) return;
  bool big = false;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < vecs; i += stride) {
    d0[i] = bf16x8_to_f16(s0[i], big);
    if (s1) d1[i] = bf16x8_to_f16(s1[i], big);
    if (s2) d2[i] = bf16x8_to_f16(s2[i], big);
  }
  if (big) set_status(status, TWELL_ERR_RANGE);
}

cudaError_t launch_to_f16(const void *const src[3], void *const dst[3], size_t elems,
                          const Ctl *ctl, int32_t *status, cudaStream_t s) {
  // (usually idle: one wave that returns when no row takes the dense path)
  launch_k(to_f16_kernel, 4 * num_sms(), 256, 0, s, (const uint4 *)src[0], (uint4 *)dst[0],
           (const uint4 *)src[1], (uint4 *)dst[1], (const uint4 *)src[2], (uint4 *)dst[2],
           elems / 8, ctl, status);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep_rows(const BwdArgs &a, cudaStream_t s) {
  const int blocks = a.T < 2 * num_sms() ? a.T : 2 * num_sms();
  launch_k(bwd_prep_rows_kernel, blocks, 256, 0, s, a.ws.ctl, a.ws.rows, (const uint4 *)a.dy,
           (const uint4 *)a.x, (uint4 *)a.ws.dyg, (uint4 *)a.ws.xg, a.D * 2 / 16, a.tw.status);
  return cudaGetLastError();
}

}  // namespace twell

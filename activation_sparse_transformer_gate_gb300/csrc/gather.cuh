// gather.cuh -- helpers of the row-gather kernels (one CTA per token or per
// neuron, 16-byte vectors of a d_model row per thread).
#pragma once

#include "common.cuh"

namespace twell {

constexpr int LIST_CAP = 2048;  // (neuron, value) pairs staged per tile group
constexpr int PB = 8;           // pairs consumed per batch
// Slot code of a no-op pair (gate 0) that pads a dense tile whose positive
// values are fewer than its count; consumers write nothing for it.
constexpr int PAD_SLOT = -2147483647 - 1;

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

// Gather NB rows (neurons s_n[b0 .. b0+nb)) of a [F][D] matrix: this thread's
// 16-byte vectors of each row, as 128-bit read-only loads that skip L1.
// Rows are `stride` vectors apart; `len` vectors are read from each row,
// starting at `base` (a column range of the rows: base is offset by the
// range's first vector, len its width).  NTH == 0: any block size; vectors
// past len and rows b >= nb (nb may be 0) are zero.  NTH > 0: a full batch
// (nb == NB) of exact rows, len = VPT * NTH vectors each, in a block of NTH
// threads: constant offsets, no predicates.
template <class T, int VPT, int NB = PB, int NTH = 0>
__device__ __forceinline__ void gather8(const uint4 *base, const int *s_n, int b0, int nb,
                                        int stride, int len, uint4 (&r)[NB][VPT]) {
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (NTH > 0) {
      const uint4 *row = base + (size_t)s_n[b0 + b] * stride + threadIdx.x;
#pragma unroll
      for (int v = 0; v < VPT; ++v) r[b][v] = ldg_stream(row + v * NTH);
    } else {
      const uint4 *row = base + (size_t)s_n[b < nb ? b0 + b : 0] * stride + threadIdx.x;  // b0 may lie past the list
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int vi = threadIdx.x + v * blockDim.x;
        r[b][v] = (b < nb && vi < len) ? ldg_stream(row + v * blockDim.x) : make_uint4(0, 0, 0, 0);
      }
    }
  }
}

// acc[0 .. EV/2) += h * (the EV values of a 16-byte vector), as packed fp32
// pair FMAs (one instruction per two products).
template <class T>
__device__ __forceinline__ void axpy_vec(float2 *acc, float h, const uint4 &w) {
  constexpr int EV = Vec<T>::EV;
  float f[EV];
  Vec<T>::unpack(w, f);
  const float2 hh = make_float2(h, h);
#pragma unroll
  for (int q = 0; q < EV / 2; ++q) acc[q] = __ffma2_rn(hh, make_float2(f[2 * q], f[2 * q + 1]), acc[q]);
}

// c + a.lo * b.lo + a.hi * b.hi for bf16 pairs packed in 32-bit words: fused
// multiply-adds with bf16 operands and an fp32 accumulator (the bf16 product
// is exact in fp32, so each step equals fmaf on the widened operands).
__device__ __forceinline__ float dot2_bf16(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %3;\n\t"
      "fma.rn.f32.bf16 %0, ah, bh, %0;}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

// ---- warp-level rows: lane l owns the 16-byte vectors l, l+32, ... of a row
// (VPL = ceil(NV / 32) of them).  A warp reduces its own dot products with
// shuffles, so pairs handled by different warps need no CTA barrier.
// EXACT: the row is exactly 32 * VPL vectors (constant offsets, no vector
// predicates); an invalid row is then left unloaded (its result is discarded).
template <int VPL, int POL = L2_NORMAL, bool EXACT = false>
__device__ __forceinline__ void warp_row(const uint4 *row, int NV, bool valid, uint4 (&r)[VPL]) {
  const int lane = threadIdx.x & 31;
  if (EXACT) {
    if (valid) {
#pragma unroll
      for (int k = 0; k < VPL; ++k) r[k] = ldg_stream<POL>(row + lane + 32 * k);
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < VPL; ++k) {
    const int vi = lane + 32 * k;
    r[k] = (valid && vi < NV) ? ldg_stream<POL>(row + vi) : make_uint4(0, 0, 0, 0);
  }
}

// Full dot product of two rows held as lane slices (warp-wide sum; every
// lane gets the result).  Two accumulator chains per lane.
template <class T, int VPL>
__device__ __forceinline__ float warp_dot(const uint4 (&a)[VPL], const uint4 (&b)[VPL]) {
  float s0 = 0.f, s1 = 0.f;
  if constexpr (Vec<T>::EV == 8) {  // bf16: mixed-precision FMAs, no widening
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      s0 = dot2_bf16(a[k].x, b[k].x, s0);
      s1 = dot2_bf16(a[k].y, b[k].y, s1);
      s0 = dot2_bf16(a[k].z, b[k].z, s0);
      s1 = dot2_bf16(a[k].w, b[k].w, s1);
    }
  } else {
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      s0 = fmaf(__uint_as_float(a[k].x), __uint_as_float(b[k].x), s0);
      s1 = fmaf(__uint_as_float(a[k].y), __uint_as_float(b[k].y), s1);
      s0 = fmaf(__uint_as_float(a[k].z), __uint_as_float(b[k].z), s0);
      s1 = fmaf(__uint_as_float(a[k].w), __uint_as_float(b[k].w), s1);
    }
  }
  float s = s0 + s1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// warp_dot with the first operand read from shared memory vector by vector
// (lane l reads vectors l, l+32, ...; zero past NV), so it holds no
// registers across the row loads.
template <class T, int VPL>
__device__ __forceinline__ float warp_dot_smem(const uint4 *s_a, int NV, const uint4 (&b)[VPL]) {
  const int lane = threadIdx.x & 31;
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int k = 0; k < VPL; ++k) {
    const int vi = lane + 32 * k;
    const uint4 a = vi < NV ? s_a[vi] : make_uint4(0, 0, 0, 0);
    if constexpr (Vec<T>::EV == 8) {
      s0 = dot2_bf16(a.x, b[k].x, s0);
      s1 = dot2_bf16(a.y, b[k].y, s1);
      s0 = dot2_bf16(a.z, b[k].z, s0);
      s1 = dot2_bf16(a.w, b[k].w, s1);
    } else {
      s0 = fmaf(__uint_as_float(a.x), __uint_as_float(b[k].x), s0);
      s1 = fmaf(__uint_as_float(a.y), __uint_as_float(b[k].y), s1);
      s0 = fmaf(__uint_as_float(a.z), __uint_as_float(b[k].z), s0);
      s1 = fmaf(__uint_as_float(a.w), __uint_as_float(b[k].w), s1);
    }
  }
  float s = s0 + s1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// warp_dot_smem without the final reduction: adds the products of vectors
// lane + 32 k (k < VPL) of s_a (zero past NV) and b into the lane's two
// partial sums, so a long row can be taken in parts with the same order of
// additions as in one piece.
template <class T, int VPL>
__device__ __forceinline__ void warp_dot_smem_acc(const uint4 *s_a, int NV, const uint4 (&b)[VPL],
                                                  float &s0, float &s1) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < VPL; ++k) {
    const int vi = lane + 32 * k;
    const uint4 a = vi < NV ? s_a[vi] : make_uint4(0, 0, 0, 0);
    if constexpr (Vec<T>::EV == 8) {
      s0 = dot2_bf16(a.x, b[k].x, s0);
      s1 = dot2_bf16(a.y, b[k].y, s1);
      s0 = dot2_bf16(a.z, b[k].z, s0);
      s1 = dot2_bf16(a.w, b[k].w, s1);
    } else {
      s0 = fmaf(__uint_as_float(a.x), __uint_as_float(b[k].x), s0);
      s1 = fmaf(__uint_as_float(a.y), __uint_as_float(b[k].y), s1);
      s0 = fmaf(__uint_as_float(a.z), __uint_as_float(b[k].z), s0);
      s1 = fmaf(__uint_as_float(a.w), __uint_as_float(b[k].w), s1);
    }
  }
}

// Where the active pairs of one (row, tile) come from.  Rows whose tiles all
// fit their K slots read the TwELL slots; an overflow row reads a dense vector
// of C ReLU values for each tile (the wide-tile buffer in the forward, the
// dense backup row in the backward) -- always (dense_all) or only for the
// tiles whose true count exceeds K.
template <class T>
struct PairSource {
  const uint8_t *idx, *nnz;
  const T *val;
  int Tn, C, K;
  int t;                 // token
  const T *dense;        // dense vector base (nullptr: slots only)
  size_t dense_tile;     // element stride between consecutive tiles' vectors
  bool dense_all;        // every tile from the dense vectors
  bool neg_slots;        // encode slots as -1 - n (results go to a dense row)
};

// Compact the pairs of tiles [g0, g0 + group) of one token into the shared
// list: s_n = neuron, s_g = gate value, s_slot = TwELL slot (or -1 - n).
// Returns the pair count.  Pairs are in ascending neuron order.  Contains
// barriers: every thread of the CTA must call it.
template <class T>
__device__ __forceinline__ int build_pairs(const PairSource<T> &ps, int g0, int group, int nt,
                                           int *s_n, float *s_g, int *s_slot, int *s_wsum,
                                           int *s_total, int32_t *status) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
  const int j = g0 + tid;
  const bool mine = tid < group && j < nt;
  const int nz = mine ? (int)ps.nnz[(size_t)j * ps.Tn + ps.t] : 0;
  const bool from_dense = mine && ps.dense && (ps.dense_all || nz > ps.K);
  const int cnt = from_dense ? nz : (nz < ps.K ? nz : ps.K);
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
    if (lane == 31) *s_total = wi;
  }
  __syncthreads();
  const int off = s_wsum[w] + incl - cnt;
  if (cnt > 0) {
    if (from_dense) {
      const T *dv = ps.dense + (size_t)j * ps.dense_tile;
      int k = 0;
      for (int c = 0; c < ps.C && k < cnt; ++c) {
        const float g = to_f(dv[c]);
        if (g > 0.f) {
          const int n = j * ps.C + c;
          s_n[off + k] = n;
          s_g[off + k] = g;
          s_slot[off + k] = -1 - n;
          ++k;
        }
      }
      for (; k < cnt; ++k) {  // fewer positive values than counted: no-op pairs
        s_n[off + k] = j * ps.C;
        s_g[off + k] = 0.f;
        s_slot[off + k] = PAD_SLOT;
      }
    } else {
      const size_t s0 = ((size_t)j * ps.Tn + ps.t) * (size_t)ps.K;
      for (int k = 0; k < cnt; ++k) {
        int c = ps.idx[s0 + k];
        if (c >= ps.C) {
          set_status(status, TWELL_ERR_INDEX);
          c = 0;
        }
        const int n = j * ps.C + c;
        s_n[off + k] = n;
        s_g[off + k] = to_f(ps.val[s0 + k]);
        s_slot[off + k] = ps.neg_slots ? -1 - n : (int)(s0 + k);
      }
    }
  }
  __syncthreads();
  return *s_total;
}

}  // namespace twell

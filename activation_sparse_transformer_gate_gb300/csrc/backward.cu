// backward.cu -- sparse backward of the TwELL FFN with the L1 term.
//
// "Sparser, Faster, Lighter Transformer Language Models", technical summary
// section 2.B (training): hybrid x dense and dense x hybrid matmuls and a sparse
// transpose for the weight gradients; L1 regularisation of the ReLU FFN
// activations.  With h = g*u (plain FFN: h = g, u = 1):
//   dh = dy . Wd[n] + lambda sign(h),  dz = [z > 0] dh u,  du = dh g
//   dx = sum_n dz Wg[n] + du Wu[n]
//   dWg[n] = sum_t dz x_t, dbg[n] = sum_t dz, dWu[n] = sum_t du x_t,
//   dWd[n] = sum_t h dy_t
// Launch sequence (on the caller's stream, except where noted):
//   1. hybrid split of the saved TwELL (overflow rows, in this workspace)
//   2. dh at the active pairs, then dz / du / h there: one CTA per token
//      from gathered W_down rows (hybrid x dense SDDMM), or, above a slot
//      density, one tensor-core GEMM dy W_down^T read at the slots; then a
//      CTA per token builds its dx row from gathered W_gate / W_up rows
//      (dense x hybrid SpMM).  Pairs come from the TwELL slots, or from the
//      dense backup row of an overflow row.  Separate passes keep each
//      pass's working set (one or two weight matrices) small enough to stay
//      in L2.
//   3. a CTA per (tile, chunk of 1024 tokens): deterministic transpose of
//      the slots into neuron-major lists ordered by token (sparse
//      transpose), from per-chunk column counts taken in step 2
//   4. one CTA per neuron: dWg, dWu, dWd rows and dbg from gathered x / dy rows
//      of its list, then the overflow rows' contributions (dense x hybrid)
// Steps 3-4 depend on step 2 only, as does the dx SpMM: they run on a second
// stream of the library, forked and joined with events, so the transpose and
// the kernels' tails overlap the SpMM (one stream while per-launch timing is
// on, so that each interval times one kernel).
#include "common.cuh"
#include "gather.cuh"
#include "kernels.h"

namespace twell {

namespace {

struct BParams {
  const void *x, *Wg, *Wu, *Wd, *dy;
  const uint8_t *idx, *nnz;
  const void *val, *u_val, *g_fb, *u_fb;
  int Tn, D, F, C, K, gated, cap;
  float lambda;
  const Ctl *ctl;
  const int32_t *rows, *pos;
  float *dz, *du, *hs;       // slot arrays [F/C][T][K]
  float *dzr, *dur, *hr;     // overflow rows [n_ovf][F]
  int32_t *col_start, *col_cnt, *col_chunk;
  float4 *col_e;             // transposed entries {token bits, dz, du, h}
  void *dx;
  float *dWg, *dbg, *dWu, *dWd;
  int gemm_rows;             // 1: the dense-path rows go through the tensor-core GEMMs
  int v0, nvp;               // dx / dW gathers: this pass's columns, in 16-byte vectors
  int32_t *status;
};

// Rows that the tensor-core GEMMs handle (every row in all-dense mode, the
// overflow rows when they take the dense GEMM path): the gather kernels skip
// them.
__device__ __forceinline__ bool gemm_row(const BParams &p, int ps) {
  return p.gemm_rows && (p.ctl->dense || (p.ctl->ovf_gemm && ps >= 0));
}

__device__ __forceinline__ float sgnf(float v) { return v > 0.f ? 1.f : (v < 0.f ? -1.f : 0.f); }

// The transpose's count of TwELL slot sl (a slot of token t, in the tile and
// column it names): col_chunk[tile][t / TR_CHUNK][column] += 1 (zeroed by the
// flags kernel at the start of the backward).  A malformed index is not
// counted, as the transpose does not list it.
__device__ __forceinline__ void count_slot(const BParams &p, int sl, int t) {
  const int c = p.idx[sl];
  if (c >= p.C) return;
  const int j = sl / (p.Tn * p.K);
  const int nch = (p.Tn + TR_CHUNK - 1) / TR_CHUNK;
  atomicAdd(&p.col_chunk[((size_t)j * nch + t / TR_CHUNK) * p.C + c], 1);
}

// Four fp32 values (two pairs) as the bit pattern of one 16-byte store.
__device__ __forceinline__ uint4 f4bits(const float2 &a, const float2 &b) {
  return make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(b.x),
                    __float_as_uint(b.y));
}

// One list entry's weight-gradient update of a thread's 16-byte column slice:
// ag += dz x, au += du x, ad += h dy (r = {token, dz, du, h}), packed fp32 pairs.
template <class T>
__device__ __forceinline__ void axpy3(float2 *ag, float2 *au, float2 *ad, const float4 &r,
                                      const uint4 &xv, const uint4 &yv) {
  constexpr int EV = Vec<T>::EV;
  float fx[EV], fy[EV];
  Vec<T>::unpack(xv, fx);
  Vec<T>::unpack(yv, fy);
  const float2 zz = make_float2(r.y, r.y), uu = make_float2(r.z, r.z), hh = make_float2(r.w, r.w);
#pragma unroll
  for (int q = 0; q < EV / 2; ++q) {
    const float2 xf = make_float2(fx[2 * q], fx[2 * q + 1]);
    ag[q] = __ffma2_rn(zz, xf, ag[q]);
    au[q] = __ffma2_rn(uu, xf, au[q]);
    ad[q] = __ffma2_rn(hh, make_float2(fy[2 * q], fy[2 * q + 1]), ad[q]);
  }
}

// ag += dz x, au += du x for one 16-byte vector of x (r = {token, dz, du, h}).
template <class T>
__device__ __forceinline__ void axpy2(float2 *ag, float2 *au, const float4 &r, const uint4 &xv) {
  constexpr int EV = Vec<T>::EV;
  float fx[EV];
  Vec<T>::unpack(xv, fx);
  const float2 zz = make_float2(r.y, r.y), uu = make_float2(r.z, r.z);
#pragma unroll
  for (int q = 0; q < EV / 2; ++q) {
    const float2 xf = make_float2(fx[2 * q], fx[2 * q + 1]);
    ag[q] = __ffma2_rn(zz, xf, ag[q]);
    au[q] = __ffma2_rn(uu, xf, au[q]);
  }
}

}  // namespace

// Pair list of one token for the backward: slots for a non-overflow row, the
// dense backup row (g_fb) for an overflow row (slot encoded as -1 - n).
template <class T>
__device__ __forceinline__ PairSource<T> bwd_source(const BParams &p, int t, int ps) {
  PairSource<T> src;
  src.idx = p.idx; src.nnz = p.nnz; src.val = (const T *)p.val; src.Tn = p.Tn; src.C = p.C;
  src.K = p.K; src.t = t;
  src.dense = ps >= 0 ? (const T *)p.g_fb + (size_t)ps * p.F : nullptr;
  src.dense_tile = p.C;
  src.dense_all = true;
  src.neg_slots = ps >= 0;
  return src;
}

// The pair's gradients from its dot d = dy . W_down[n]: dh = d + lambda
// sign(h), dz = [g > 0] dh u, du = [g > 0] dh g, and h = g u (plain FFN:
// u = 1), stored at the TwELL slot (sl >= 0) or in the overflow-row arrays
// (sl = -1 - n).  Pad pairs (PAD_SLOT) store nothing.
template <class T>
__device__ __forceinline__ void dh_finish(const BParams &p, int ps, int sl, float g, float d) {
  if (sl == PAD_SLOT) return;
  const float u = !p.gated ? 1.f
                           : (sl >= 0 ? to_f(((const T *)p.u_val)[sl])
                                      : to_f(((const T *)p.u_fb)[(size_t)ps * p.F + (-1 - sl)]));
  const float h = p.gated ? g * u : g;
  const float dh = d + p.lambda * sgnf(h);
  const bool act = g > 0.f;
  const float dz = act ? (p.gated ? dh * u : dh) : 0.f;
  const float du = act ? dh * g : 0.f;
  if (sl >= 0) {
    p.dz[sl] = dz;
    p.du[sl] = du;
    p.hs[sl] = h;
    count_slot(p, sl, (sl / p.K) % p.Tn);
  } else {
    const size_t o = (size_t)ps * p.F + (-1 - sl);
    p.dzr[o] = dz;
    p.dur[o] = du;
    p.hr[o] = h;
  }
}

// ---------------------------------------------------------------------------
// 2a. Per-token dh SDDMM (hybrid x dense): dh = dy . Wd[n] + lambda sign(h) at
// every active pair, then dz, du, h of the pair -- at its TwELL slot for a
// non-overflow row, in the overflow-row arrays for an overflow row.  Only
// W_down rows are gathered, so the working set is W_down and dy.  Each warp
// computes whole dot products for its share of the pairs (PIF rows in flight,
// warp shuffles only): no barrier inside the pair loop.  One row per warp,
// with dy read from shared memory inside the dot, fits 64 registers at
// d_model <= 2048 (four CTAs per SM), which hides more latency than a second
// row per warp.
template <class T, int VL, int PIF>
__global__ void __launch_bounds__(256, VL <= 8 ? 4 : 2) bwd_dh_kernel(BParams p) {
  pdl_begin();
  constexpr int EV = Vec<T>::EV;
  __shared__ int s_n[LIST_CAP];
  __shared__ float s_g[LIST_CAP];
  __shared__ int s_slot[LIST_CAP];
  __shared__ uint4 s_dy[1024];
  __shared__ int s_wsum[32];
  __shared__ int s_total;

  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nw = blockDim.x >> 5;
  const int nt = p.F / p.C;
  const int NV = p.D / EV;
  if (p.ctl->dh_gemm) return;  // dh came from the tensor-core GEMM
  const int ps = p.pos[t];
  if (ps >= p.cap) return;  // overflow row without a dense backup row (capacity error)
  if (gemm_row(p, ps)) return;
  for (int v = tid; v < NV; v += blockDim.x) s_dy[v] = ((const uint4 *)p.dy)[(size_t)t * NV + v];
  const uint4 *Wd4 = (const uint4 *)p.Wd;
  const PairSource<T> src = bwd_source<T>(p, t, ps);
  int group = LIST_CAP / (ps >= 0 ? p.C : p.K);
  if (group > (int)blockDim.x) group = blockDim.x;
  for (int g0 = 0; g0 < nt; g0 += group) {
    const int P = build_pairs(src, g0, group, nt, s_n, s_g, s_slot, s_wsum, &s_total, p.status);
    for (int i0 = w; i0 < P; i0 += nw * PIF) {
      uint4 wr[PIF][VL];
#pragma unroll
      for (int q = 0; q < PIF; ++q) {
        const int i = i0 + q * nw;
        warp_row<VL>(Wd4 + (size_t)s_n[i < P ? i : i0] * NV, NV, i < P, wr[q]);
      }
#pragma unroll
      for (int q = 0; q < PIF; ++q) {
        const int i = i0 + q * nw;
        const float d = warp_dot_smem<T, VL>(s_dy, NV, wr[q]);
        if (lane == 0 && i < P) dh_finish<T>(p, ps, s_slot[i], s_g[i], d);
      }
    }
    __syncthreads();  // the list is rewritten by the next group
  }
}

// ---------------------------------------------------------------------------
// 2a'. The same dh SDDMM on the tensor cores (bf16, d_model a multiple of 256).
// One CTA (8 warps) per token; the pairs are taken 16 at a time, and warp w
// covers the w-th eighth of d_model for all 16: per 32-element chunk one
// mma.sync.m16n8k16 pair with A = the 16 gathered W_down rows (thread (g, q)
// loads 16 bytes of rows g and g + 8) and B = the dy chunk in column 0 (lanes
// 0-3; the other columns are zero).  A and B take the chunk's elements in the
// same order, so C[r][0] is the partial dot of row r.  The eight partials of
// a pair are summed in a fixed order in shared memory, then one thread per
// pair applies dh_finish.  The tensor core does the multiply-adds and the
// reduction that the warp-level kernel spends most of its instructions on.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
      " {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int DH_WARPS = 8;
constexpr int DH_CHUNK = 256;  // pairs whose partial dots are held before the finish

// WIDE (U even, W_down 32-byte aligned): lane q of a row group takes the
// 32 contiguous bytes (vectors 2q, 2q + 1) of each pair of chunks in one
// 256-bit load, so one load instruction covers 128 contiguous bytes of each
// of its 8 rows -- half the L1 wavefronts of four lanes x 16 bytes -- and dy
// is read at the same vectors.
template <int U, bool WIDE>
__global__ void __launch_bounds__(DH_WARPS * 32, U >= 8 ? 2 : (U >= 4 ? 3 : 4))
    bwd_dh_mma_kernel(BParams p) {
  pdl_begin();
  __shared__ int s_n[LIST_CAP];
  __shared__ float s_g[LIST_CAP];
  __shared__ int s_slot[LIST_CAP];
  __shared__ uint4 s_dy[1024];
  __shared__ float s_u[DH_CHUNK];
  __shared__ float s_part[DH_WARPS][DH_CHUNK];
  __shared__ int s_wsum[32];
  __shared__ int s_total;

  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int gq = lane >> 2, q = lane & 3;
  const int nt = p.F / p.C;
  const int NV = p.D / 8;               // 16-byte vectors per row
  const int CPW = NV / (4 * DH_WARPS);  // 32-element chunks per warp (NV % 32 == 0)
  if (p.ctl->dh_gemm) return;  // dh came from the tensor-core GEMM
  const int ps = p.pos[t];
  if (ps >= p.cap) return;  // overflow row without a dense backup row (capacity error)
  if (gemm_row(p, ps)) return;
  for (int v = tid; v < NV; v += blockDim.x) s_dy[v] = ((const uint4 *)p.dy)[(size_t)t * NV + v];
  const uint4 *Wd4 = (const uint4 *)p.Wd;
  // this lane's dy vectors (read by lanes 0-3)
  const uint4 *dyw = s_dy + 4 * w * CPW + (WIDE ? 2 * q : q);
  const bf16 *uval = (const bf16 *)p.u_val, *ufb = (const bf16 *)p.u_fb;
  const PairSource<bf16> src = bwd_source<bf16>(p, t, ps);
  int group = LIST_CAP / (ps >= 0 ? p.C : p.K);
  if (group > (int)blockDim.x) group = blockDim.x;
  for (int g0 = 0; g0 < nt; g0 += group) {
    const int P = build_pairs(src, g0, group, nt, s_n, s_g, s_slot, s_wsum, &s_total, p.status);
    for (int cb = 0; cb < P; cb += DH_CHUNK) {
      const int PC = P - cb < DH_CHUNK ? P - cb : DH_CHUNK;
      // u of the chunk's pairs, fetched while the rows stream in
      if (tid < PC) {
        const int sl = s_slot[cb + tid];
        s_u[tid] = (!p.gated || sl == PAD_SLOT) ? 1.f
                   : to_f(sl >= 0 ? uval[sl] : ufb[(size_t)ps * p.F + (-1 - sl)]);
      }
      for (int pb = 0; pb < PC; pb += 16) {
        // rows g and g + 8 of the block (past the chunk: its first row, result unused)
        const int r0 = pb + gq < PC ? pb + gq : pb, r1 = pb + gq + 8 < PC ? pb + gq + 8 : pb;
        const int lq = WIDE ? 2 * q : q;
        const uint4 *w0 = Wd4 + (size_t)s_n[cb + r0] * NV + 4 * w * CPW + lq;
        const uint4 *w1 = Wd4 + (size_t)s_n[cb + r1] * NV + 4 * w * CPW + lq;
        // two accumulator chains (even / odd half of each chunk)
        float c[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c0 = 0; c0 < CPW; c0 += U) {
          uint4 A0[U], A1[U];
          if (WIDE) {  // chunks (c0 + 2v, c0 + 2v + 1): vectors 8v + 2q, 8v + 2q + 1
#pragma unroll
            for (int v = 0; v < U / 2; ++v) {
              ldg_stream32(w0 + 4 * c0 + 8 * v, A0[2 * v], A0[2 * v + 1]);
              ldg_stream32(w1 + 4 * c0 + 8 * v, A1[2 * v], A1[2 * v + 1]);
            }
          } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
              A0[u] = ldg_stream(w0 + 4 * (c0 + u));
              A1[u] = ldg_stream(w1 + 4 * (c0 + u));
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int dv = WIDE ? 4 * c0 + 8 * (u >> 1) + (u & 1) : 4 * (c0 + u);
            const uint4 b = gq == 0 ? dyw[dv] : make_uint4(0, 0, 0, 0);
            mma_bf16_16816(c, A0[u].x, A1[u].x, A0[u].y, A1[u].y, b.x, b.y);
            mma_bf16_16816(e, A0[u].z, A1[u].z, A0[u].w, A1[u].w, b.z, b.w);
          }
        }
        if (q == 0) {  // C[g][0] and C[g + 8][0]
          if (pb + gq < PC) s_part[w][pb + gq] = c[0] + e[0];
          if (pb + gq + 8 < PC) s_part[w][pb + gq + 8] = c[2] + e[2];
        }
      }
      __syncthreads();
      if (tid < PC) {  // one thread per pair: partials in a fixed order
        float d = 0.f;
#pragma unroll
        for (int k = 0; k < DH_WARPS; ++k) d += s_part[k][tid];
        const int i = cb + tid, sl = s_slot[i];
        if (sl != PAD_SLOT) {
          const float g = s_g[i], u = s_u[tid];
          const float h = p.gated ? g * u : g;
          const float dh = d + p.lambda * sgnf(h);
          const bool act = g > 0.f;
          const float dz = act ? (p.gated ? dh * u : dh) : 0.f;
          const float du = act ? dh * g : 0.f;
          if (sl >= 0) {
            p.dz[sl] = dz;
            p.du[sl] = du;
            p.hs[sl] = h;
            count_slot(p, sl, t);
          } else {
            const size_t o = (size_t)ps * p.F + (-1 - sl);
            p.dzr[o] = dz;
            p.dur[o] = du;
            p.hr[o] = h;
          }
        }
      }
      __syncthreads();  // s_part / s_u are rewritten by the next chunk
    }
  }
}

// ---------------------------------------------------------------------------
// 2b. Per-token dx SpMM (dense x hybrid): dx_t = sum over active pairs of
// dz W_gate[n] + du W_up[n].  No reductions, no barriers in the pair loop;
// the working set is W_gate and W_up, or the column range [v0, v0 + nvp)
// of both when the launch is split into column passes (each element of dx
// sums the same products in the same order either way).
template <class T, int VPT, int NB, int NTH>
__global__ void __launch_bounds__(256) bwd_dx_kernel(BParams p) {
  pdl_begin();
  constexpr int EV = Vec<T>::EV;
  __shared__ int s_n[LIST_CAP];
  __shared__ float s_g[LIST_CAP];
  __shared__ float s_z[LIST_CAP];
  __shared__ float s_u[LIST_CAP];
  __shared__ int s_slot[LIST_CAP];
  __shared__ int s_wsum[32];
  __shared__ int s_total;

  const int t = blockIdx.x, tid = threadIdx.x;
  const int nt = p.F / p.C;
  const int NV = p.D / EV;             // row stride
  const int v0 = p.v0, NP = p.nvp;     // this pass's vectors of each row
  const int ps = p.pos[t];
  if (ps >= p.cap || gemm_row(p, ps)) return;
  float2 dxg[VPT][EV / 2], dxu[VPT][EV / 2];  // two accumulator chains
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int e = 0; e < EV / 2; ++e) dxg[v][e] = dxu[v][e] = make_float2(0.f, 0.f);
  const uint4 *Wg4 = (const uint4 *)p.Wg + v0;
  const uint4 *Wu4 = p.gated ? (const uint4 *)p.Wu + v0 : nullptr;
  const PairSource<T> src = bwd_source<T>(p, t, ps);
  int group = LIST_CAP / (ps >= 0 ? p.C : p.K);
  if (group > (int)blockDim.x) group = blockDim.x;
  for (int g0 = 0; g0 < nt; g0 += group) {
    const int P = build_pairs(src, g0, group, nt, s_n, s_g, s_slot, s_wsum, &s_total, p.status);
    for (int i = tid; i < P; i += blockDim.x) {
      const int sl = s_slot[i];
      if (sl == PAD_SLOT) {
        s_z[i] = 0.f;
        s_u[i] = 0.f;
        continue;
      }
      const size_t o = (size_t)ps * p.F + (-1 - sl);
      s_z[i] = sl >= 0 ? p.dz[sl] : p.dzr[o];
      s_u[i] = sl >= 0 ? p.du[sl] : p.dur[o];
    }
    __syncthreads();
    for (int b0 = 0; b0 < P; b0 += NB) {
      const int nb = P - b0 < NB ? P - b0 : NB;
      uint4 wg[NB][VPT], wu[NB][VPT];
      if (NTH > 0 && nb == NB) {
        gather8<T, VPT, NB, NTH>(Wg4, s_n, b0, nb, NV, NP, wg);
        if (p.gated) gather8<T, VPT, NB, NTH>(Wu4, s_n, b0, nb, NV, NP, wu);
      } else {
        gather8<T, VPT, NB>(Wg4, s_n, b0, nb, NV, NP, wg);
        if (p.gated) gather8<T, VPT, NB>(Wu4, s_n, b0, nb, NV, NP, wu);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= nb) break;
        const float z = s_z[b0 + b], u = s_u[b0 + b];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          axpy_vec<T>(dxg[v], z, wg[b][v]);
          if (p.gated) axpy_vec<T>(dxu[v], u, wu[b][v]);
        }
      }
    }
    __syncthreads();
  }
  uint4 *dxrow = (uint4 *)p.dx + (size_t)t * NV + v0;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int vi = tid + v * blockDim.x;
    float o[EV];
#pragma unroll
    for (int e = 0; e < EV / 2; ++e) {
      o[2 * e] = dxg[v][e].x + dxu[v][e].x;
      o[2 * e + 1] = dxg[v][e].y + dxu[v][e].y;
    }
    if (vi < NP) stg_stream(dxrow + vi, Vec<T>::pack(o));
  }
}

// ---------------------------------------------------------------------------
// 3. Sparse transpose of the slots into neuron-major lists.  The list of
// neuron j*C + c occupies col_e[col_start .. + col_cnt) inside tile j's region
// [j*T*K, (j+1)*T*K), ordered by token; each entry carries the token and the
// pair's dz, du, h, so the weight-gradient pass reads one 16-byte record per
// entry.  Overflow rows are not listed (their pairs live in the overflow-row
// arrays).  The entries of every column in each chunk of 1024 tokens were
// counted by the dh kernels (count_slot); one pass over a (tile, chunk) grid
// then places them: the chunk's first entry per column = the column's start
// in the tile (prefix over columns of the totals) + the counts of earlier
// chunks; a token's rank among the chunk's tokens that use column c comes
// from per-warp lane masks (popc below the lane) plus per-warp offsets.
template <int C>
__global__ void __launch_bounds__(TR_CHUNK) twell_transpose_kernel(BParams p) {
  pdl_begin();
  __shared__ uint32_t occ[32][C];
  __shared__ int woff[32][C];
  __shared__ int run[C], tot[C];
  __shared__ int wsum[32];
  const int j = blockIdx.x, ch = blockIdx.y, nch = gridDim.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int K = p.K, Tn = p.Tn;
  const size_t region = (size_t)j * Tn * K;
  const int32_t *cc = p.col_chunk + (size_t)j * nch * C;
  // per column: entries of earlier chunks and of all chunks
  for (int c = tid; c < C; c += blockDim.x) {
    int before = 0, all = 0;
    for (int q = 0; q < nch; ++q) {
      const int v = cc[(size_t)q * C + c];
      all += v;
      if (q < ch) before += v;
    }
    run[c] = before;
    tot[c] = all;
  }
  for (int i = tid; i < 32 * C; i += blockDim.x) (&occ[0][0])[i] = 0u;
  __syncthreads();
  // exclusive prefix of the column totals (C <= 128: four warps of 32)
  if (tid < C) {
    const int v = tot[tid];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[w] = incl;
    tot[tid] = incl - v;  // exclusive within the warp for now
  }
  __syncthreads();
  if (tid < C) {
    int off = 0;
    for (int q = 0; q < w; ++q) off += wsum[q];
    const int start = tot[tid] + off;
    run[tid] += start;
    if (ch == 0) {
      p.col_start[j * C + tid] = (int)(region + start);
      int all = 0;
      for (int q = 0; q < nch; ++q) all += cc[(size_t)q * C + tid];
      p.col_cnt[j * C + tid] = all;
    }
  }
  const unsigned lt = (1u << lane) - 1u;
  const int t = ch * TR_CHUNK + tid;
  const bool act = t < Tn && p.pos[t] < 0 && !(p.gemm_rows && p.ctl->dense);
  const int n = act ? (int)p.nnz[(size_t)j * Tn + t] : 0;
  const size_t s0 = ((size_t)j * Tn + (act ? t : 0)) * K;
  for (int k = 0; k < n && k < K; ++k) {
    const int c = p.idx[s0 + k];
    if (c < C) atomicOr(&occ[w][c], 1u << lane);
  }
  __syncthreads();
  for (int c = tid; c < C; c += blockDim.x) {
    int r = run[c];
    for (int q = 0; q < 32; ++q) {
      woff[q][c] = r;
      r += __popc(occ[q][c]);
    }
  }
  __syncthreads();
  for (int k = 0; k < n && k < K; ++k) {
    const int c = p.idx[s0 + k];
    if (c >= C) continue;
    const int e = woff[w][c] + __popc(occ[w][c] & lt);
    const size_t sl = s0 + k;
    p.col_e[region + e] = make_float4(__int_as_float(t), p.dz[sl], p.du[sl], p.hs[sl]);
  }
}

// ---------------------------------------------------------------------------
// 4. One CTA per neuron: weight-gradient rows from the neuron's list
// (ascending tokens), then the overflow rows (ascending).  Rows of neurons
// that are never active are written as zeros.  The list is staged in shared
// memory first (one coalesced load), so each batch of PB tokens costs one
// round trip: its x and dy rows.  Split into column passes, a CTA handles
// the columns [v0, v0 + nvp) of the neuron's rows (the working set is that
// range of x and dy; every element sums the same products in the same
// order); dbg is written by the first pass.
constexpr int DW_LIST = 512;

// PART 0: all three gradients; 1: dW_gate, dW_up and dbg (x rows only); 2:
// dW_down (dy rows only).  Split in two, each launch gathers one matrix's
// rows (half the working set) and holds fewer accumulators, so it needs
// fewer registers per thread and more CTAs fit on an SM (86 and 63 against
// 128 registers at d_model 2048).  Measured: x + dy of 134 MB (d_model 2048
// at 16384 tokens; d_model 4096 at 8192) 0.735 -> 0.686 ms and 0.739 ->
// 0.706 ms; at 34 MB (d_model 2048, 4096 tokens) it loses, 0.211 -> 0.222
// ms (each part repeats the per-neuron list staging and row stores), so
// the split is taken only when x + dy exceed half of L2.
template <class T, int VPT, int NB, int NTH, int PART>
__global__ void __launch_bounds__(256) bwd_dw_kernel(BParams p) {
  pdl_begin();
  constexpr int EV = Vec<T>::EV;
  constexpr bool DX = PART != 2, DY = PART != 1;  // x rows (dW_gate, dW_up) / dy rows (dW_down)
  __shared__ float4 s_e[DW_LIST];
  if (p.gemm_rows && p.ctl->dense) return;  // the GEMMs write every row
  const int n = blockIdx.x, tid = threadIdx.x;
  const int NV = p.D / EV;             // row stride
  const int v0 = p.v0, NP = p.nvp;     // this pass's vectors of each row
  const uint4 *x4 = (const uint4 *)p.x + v0, *dy4 = (const uint4 *)p.dy + v0;
  float2 ag[VPT][EV / 2], au[VPT][EV / 2], ad[VPT][EV / 2];
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int e = 0; e < EV / 2; ++e) ag[v][e] = au[v][e] = ad[v][e] = make_float2(0.f, 0.f);
  float sb = 0.f;
  const int start = p.col_start[n], cnt = p.col_cnt[n];
  for (int c0 = 0; c0 < cnt; c0 += DW_LIST) {
    const int m = cnt - c0 < DW_LIST ? cnt - c0 : DW_LIST;
    if (c0) __syncthreads();  // the previous chunk is consumed
    for (int i = tid; i < m; i += blockDim.x) s_e[i] = p.col_e[start + c0 + i];
    __syncthreads();
    for (int e0 = 0; e0 < m; e0 += NB) {
      const int nb = m - e0 < NB ? m - e0 : NB;
      uint4 xv[NB][VPT], yv[NB][VPT];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int t = __float_as_int(s_e[e0 + (b < nb ? b : 0)].x);
        const uint4 *xr = x4 + (size_t)t * NV + tid, *yr = dy4 + (size_t)t * NV + tid;
        if (NTH > 0 && nb == NB) {  // full batch of exact rows: constant offsets
#pragma unroll
          for (int v = 0; v < VPT; ++v) {
            if (DX) xv[b][v] = ldg_stream(xr + v * NTH);
            if (DY) yv[b][v] = ldg_stream(yr + v * NTH);
          }
        } else {
#pragma unroll
          for (int v = 0; v < VPT; ++v) {
            const int vi = tid + v * blockDim.x;
            const bool ok = b < nb && vi < NP;
            if (DX) xv[b][v] = ok ? ldg_stream(xr + v * blockDim.x) : make_uint4(0, 0, 0, 0);
            if (DY) yv[b][v] = ok ? ldg_stream(yr + v * blockDim.x) : make_uint4(0, 0, 0, 0);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= nb) break;
        const float4 r = s_e[e0 + b];
        sb += r.y;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          if (DX && DY) axpy3<T>(ag[v], au[v], ad[v], r, xv[b][v], yv[b][v]);
          else if (DX) axpy2<T>(ag[v], au[v], r, xv[b][v]);
          else axpy_vec<T>(ad[v], r.w, yv[b][v]);
        }
      }
    }
  }
  // overflow rows (dense backup), unless the GEMMs add them afterwards
  const int n_rows = (p.gemm_rows && p.ctl->ovf_gemm) ? 0 : min(p.ctl->n_ovf, p.cap);
  const T *gfb = (const T *)p.g_fb;
  for (int i = 0; i < n_rows; ++i) {
    if (!(to_f(gfb[(size_t)i * p.F + n]) > 0.f)) continue;
    const int t = p.rows[i];
    const float4 r = make_float4(0.f, p.dzr[(size_t)i * p.F + n], p.dur[(size_t)i * p.F + n],
                                 p.hr[(size_t)i * p.F + n]);
    sb += r.y;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int vi = tid + v * blockDim.x;
      if (vi >= NP) continue;
      if (DX && DY) axpy3<T>(ag[v], au[v], ad[v], r, x4[(size_t)t * NV + vi], dy4[(size_t)t * NV + vi]);
      else if (DX) axpy2<T>(ag[v], au[v], r, x4[(size_t)t * NV + vi]);
      else axpy_vec<T>(ad[v], r.w, dy4[(size_t)t * NV + vi]);
    }
  }
  const size_t o0 = (size_t)n * p.D + (size_t)v0 * EV;
  float4 *og = (float4 *)(p.dWg + o0), *od = (float4 *)(p.dWd + o0);
  float4 *ou = p.gated ? (float4 *)(p.dWu + o0) : nullptr;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int vi = tid + v * blockDim.x;
    if (vi >= NP) continue;
#pragma unroll
    for (int q = 0; q < EV / 4; ++q) {
      if (DX) stg_stream(og + vi * (EV / 4) + q, f4bits(ag[v][2 * q], ag[v][2 * q + 1]));
      if (DY) stg_stream(od + vi * (EV / 4) + q, f4bits(ad[v][2 * q], ad[v][2 * q + 1]));
      if (DX && ou) stg_stream(ou + vi * (EV / 4) + q, f4bits(au[v][2 * q], au[v][2 * q + 1]));
    }
  }
  if (DX && tid == 0 && v0 == 0) p.dbg[n] = sb;
}

// ---------------------------------------------------------------------------
cudaError_t aux_stream(AuxStream *&out) {
  static thread_local AuxStream per_dev[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  AuxStream &a = per_dev[dev];
  if (!a.s2) {
    e = cudaStreamCreateWithFlags(&a.s2, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&a.s3, cudaStreamNonBlocking);
    for (cudaEvent_t *ev : {&a.fork, &a.join, &a.fork3, &a.join3, &a.mid})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {  // release what was made; the next call tries again
      for (cudaEvent_t *ev : {&a.mid, &a.join3, &a.fork3, &a.join, &a.fork}) {
        if (*ev) cudaEventDestroy(*ev);
        *ev = nullptr;
      }
      if (a.s3) cudaStreamDestroy(a.s3);
      if (a.s2) cudaStreamDestroy(a.s2);
      a.s2 = a.s3 = nullptr;
      return e;
    }
  }
  out = &a;
  return cudaSuccess;
}

cudaError_t launch_backward(const BwdArgs &a, cudaStream_t s) {
  BParams p;
  p.x = a.x; p.Wg = a.Wg; p.Wu = a.Wu; p.Wd = a.Wd; p.dy = a.dy;
  p.idx = a.tw.idx; p.nnz = a.tw.nnz; p.val = a.tw.val; p.u_val = a.tw.u_val;
  p.g_fb = a.tw.g_fb; p.u_fb = a.tw.u_fb;
  p.Tn = a.T; p.D = a.D; p.F = a.F; p.C = a.C; p.K = a.K; p.gated = a.gated;
  p.cap = a.tw.ovf_cap; p.lambda = a.lambda;
  p.ctl = a.ws.ctl; p.rows = a.ws.rows; p.pos = a.ws.pos;
  p.dz = a.ws.dz; p.du = a.ws.du; p.hs = a.ws.hs;
  p.dzr = a.ws.dzr; p.dur = a.ws.dur; p.hr = a.ws.hr;
  p.col_start = a.ws.col_ptr; p.col_cnt = a.ws.col_cnt; p.col_e = a.ws.col_e; p.col_chunk = a.ws.col_chunk;
  p.dx = a.dx; p.dWg = a.dWg; p.dbg = a.dbg; p.dWu = a.dWu; p.dWd = a.dWd;
  p.status = a.tw.status;
  const bool bf = a.dtype == TWELL_BF16;
  const bool tc = bf && tc_available();
  // the dense-path rows' tensor-core GEMMs (when the workspace has their buffers)
  const bool gemm = tc && a.ws.dense_bufs;
  p.gemm_rows = gemm ? 1 : 0;
  p.v0 = 0;
  p.nvp = a.D / (bf ? 8 : 4);

  // 1. hybrid split of the saved activations into this workspace, with the
  // forward's dispatcher rules when the dense-path rows have GEMMs
  prof_mark(KID_START, s);
  cudaError_t e = launch_flags_from_nnz(a.tw, a.ws.ovf_bits, a.ws.slot_parts, s, a.ws.col_chunk,
                                        a.F * ((a.T + TR_CHUNK - 1) / TR_CHUNK));
  if (e != cudaSuccess) return e;
  e = launch_overflow_compact(a.tw, &a.ws, gemm ? a.dense_switch : 2.0f, s, /*write_user=*/false,
                              gemm ? a.dense_density : -1.f, a.ws.slot_parts, flags_blocks(a.T),
                              tc ? a.dh_density : -1.f);
  if (e != cudaSuccess) return e;
  prof_mark(KID_OVERFLOW_COMPACT, s, 2);
  // Side streams (the caller's stream alone while per-launch timing is on,
  // so that each interval times one kernel): s3 runs the dense-path rows'
  // chain, s2 the sparse transpose and the weight-gradient gathers.
  const bool fork = !prof_enabled();
  AuxStream *aux = nullptr;
  cudaStream_t sd = s, sw = s;
  if (fork) {
    e = aux_stream(aux);
    if (e != cudaSuccess) return e;
    sd = aux->s3;
    sw = aux->s2;
  }
  // 1'. dense-path rows on the tensor cores (idle when there are none):
  // gathered dy / x rows, dh -> dz / du / h, dx.  They own other rows (and
  // other buffers) than the gather path, so they run beside it on s3.
  bool forked3 = false;
  if (gemm) {
    if (fork) {
      e = cudaEventRecord(aux->fork3, s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(sd, aux->fork3, 0);
      if (e != cudaSuccess) return e;
      forked3 = true;
    }
    e = launch_bwd_prep_rows(a, sd);
    if (e == cudaSuccess) {  // the fp16 operand copies of the weights
      prof_mark(KID_BWD_PREP, sd);
      const void *src[3] = {a.Wd, a.Wg, a.gated ? a.Wu : nullptr};
      void *const dst[3] = {a.ws.wd16, a.ws.wg16, a.gated ? a.ws.wu16 : nullptr};
      e = launch_to_f16(src, dst, (size_t)a.F * (size_t)a.D, a.ws.ctl, a.tw.status, sd);
    }
    if (e == cudaSuccess) {
      prof_mark(KID_TO_F16, sd);
      e = launch_tc_bwd_dh(a, sd);
    }
    if (e == cudaSuccess) {
      prof_mark(KID_BWD_DENSE, sd);
      e = launch_tc_bwd_dx(a, sd);
    }
    if (e == cudaSuccess) prof_mark(KID_BWD_DENSE_DX, sd);
    if (e == cudaSuccess && fork) e = cudaEventRecord(aux->mid, sd);  // dense rows' dh done
  }
  // joins s3 back into the caller's stream (also after an error)
  auto join3 = [&](cudaError_t err) {
    if (!forked3) return err;
    const cudaError_t j1 = cudaEventRecord(aux->join3, sd);
    const cudaError_t j2 = j1 == cudaSuccess ? cudaStreamWaitEvent(s, aux->join3, 0) : j1;
    return err == cudaSuccess ? j2 : err;
  };
  if (e != cudaSuccess) return join3(e);
  // 2. dh of the rows the gathers own: one tensor-core GEMM read at the
  // slots when the dispatcher chose it (its CTAs return at once otherwise),
  // else the per-token SDDMM (whose CTAs then return at once); then dx SpMM
  if (tc) {
    e = launch_tc_bwd_dh_sampled(a, s);
    if (e != cudaSuccess) return join3(e);
    prof_mark(KID_BWD_DH_GEMM, s);
  }
  const int EV = bf ? 8 : 4;
  const int NV = a.D / EV;
  const int vl = NV <= 32 ? 1 : NV <= 64 ? 2 : NV <= 128 ? 4 : NV <= 256 ? 8 : NV <= 512 ? 16 : 32;
// (the constant-offset row loads that help the SpMM kernels made this one slower)
#define TW_DH(TT, L) launch_k(bwd_dh_kernel<TT, L, 1>, a.T, 256, 0, s, p)
#define TW_DH_T(TT)                                                                            \
  do {                                                                                         \
    switch (vl) {                                                                              \
      case 1: TW_DH(TT, 1); break;                                                             \
      case 2: TW_DH(TT, 2); break;                                                             \
      case 4: TW_DH(TT, 4); break;                                                             \
      case 8: TW_DH(TT, 8); break;                                                             \
      case 16: TW_DH(TT, 16); break;                                                           \
      default: TW_DH(TT, 32); break;                                                           \
    }                                                                                          \
  } while (0)
  if (bf && NV % (4 * DH_WARPS) == 0) {
    // tensor-core dh SDDMM: chunks per warp = NV / 32; U of them per load
    // batch (4: three CTAs per SM, measured faster than 8 at two)
    const int cpw = NV / (4 * DH_WARPS);
    // 256-bit row loads need 32-byte aligned rows (the ABI promises 16)
    const bool wide = ((uintptr_t)a.Wd & 31u) == 0 && (a.D * 2) % 32 == 0;
    if (cpw % 4 == 0 && wide) launch_k(bwd_dh_mma_kernel<4, true>, a.T, DH_WARPS * 32, 0, s, p);
    else if (cpw % 4 == 0) launch_k(bwd_dh_mma_kernel<4, false>, a.T, DH_WARPS * 32, 0, s, p);
    else if (cpw % 2 == 0 && wide)
      launch_k(bwd_dh_mma_kernel<2, true>, a.T, DH_WARPS * 32, 0, s, p);
    else if (cpw % 2 == 0) launch_k(bwd_dh_mma_kernel<2, false>, a.T, DH_WARPS * 32, 0, s, p);
    else launch_k(bwd_dh_mma_kernel<1, false>, a.T, DH_WARPS * 32, 0, s, p);
  } else if (bf) {
    TW_DH_T(bf16);
  } else {
    TW_DH_T(float);
  }
#undef TW_DH_T
#undef TW_DH
  e = cudaGetLastError();
  if (e != cudaSuccess) return join3(e);
  prof_mark(KID_BWD_SLOTS, s);
  // Token / neuron CTAs over the column passes of the dx and dW gathers: each
  // thread owns two 16-byte vectors of a row (half the per-row overhead of
  // one), batches of 3 rows per matrix in flight.
  const size_t es = bf ? 2 : 4;
  const int dx_passes = gather_passes(a.tw.gather_passes, (a.gated ? 2.0 : 1.0) * a.F * a.D * es, NV,
                                      GATHER_MIN_WIDTH);
  // dW: x rows and dy rows in separate launches when together they exceed
  // half of L2 (any forced pass count > 1 splits too), and column passes
  // chosen on x + dy together (d_model 4096 at 8192 tokens: split and two
  // column passes 0.71 ms, split alone 0.82, two column passes alone 0.74)
  const double dw_set = 2.0 * a.T * a.D * es;
  const bool dw_split = a.tw.gather_passes > 0 ? a.tw.gather_passes > 1
                                               : dw_set > 0.5 * (double)l2_size();
  const int dw_passes = gather_passes(a.tw.gather_passes, dw_set, NV, GATHER_MIN_WIDTH);
// NB2: batches of two rows (instead of four) in the exact 128-thread shape:
// fewer registers, five CTAs per SM instead of four.  Measured better where
// the rows come partly from DRAM (passes over a working set beyond L2: dx
// at d_model 4096, 0.678 -> 0.659 ms) and for the split dW launches (0.707
// -> 0.672 ms at d_model 4096, 0.689 -> 0.665 at d_model 2048 / 16384
// tokens); worse at d_model 2048 / 4096 tokens (dx 0.186 -> 0.194 ms).
#define TW_VPT(K, TT, G, SS, NPASS, EXTRA, NB2)                                                \
  do {                                                                                         \
    for (int i_ = 0; i_ < (NPASS); ++i_) {                                                     \
      p.v0 = (int)((long)NV * i_ / (NPASS));                                                   \
      p.nvp = (int)((long)NV * (i_ + 1) / (NPASS)) - p.v0;                                     \
      const int np_ = p.nvp;                                                                   \
      const int vpt = np_ <= 64 ? 1 : np_ <= 512 ? 2 : 4;                                      \
      const int threads = ((np_ + vpt - 1) / vpt + 31) / 32 * 32;                              \
      if (vpt == 1) launch_k(K<TT, 1, 8, 0 EXTRA>, G, threads, 0, SS, p);                      \
      else if (vpt == 2 && np_ == 256 && (NB2)) launch_k(K<TT, 2, 2, 128 EXTRA>, G, 128, 0, SS, p); \
      else if (vpt == 2 && np_ == 256) launch_k(K<TT, 2, 4, 128 EXTRA>, G, 128, 0, SS, p);     \
      else if (vpt == 2) launch_k(K<TT, 2, 3, 0 EXTRA>, G, threads, 0, SS, p);                 \
      else launch_k(K<TT, 4, 2, 0 EXTRA>, G, threads, 0, SS, p);                               \
    }                                                                                          \
    p.v0 = 0;                                                                                  \
    p.nvp = NV;                                                                                \
  } while (0)
  // Steps 3-4 on s2: forked here, after dh, and joined before returning.
  if (fork) {
    e = cudaEventRecord(aux->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sw, aux->fork, 0);
    if (e != cudaSuccess) return join3(e);
  }
  const int nt = a.F / a.C;
  const dim3 tgrid(nt, (a.T + TR_CHUNK - 1) / TR_CHUNK);
  auto transpose = [&]() {  // 3. (the per-chunk column counts were taken with dh)
    if (a.C == 32) launch_k(twell_transpose_kernel<32>, tgrid, TR_CHUNK, 0, sw, p);
    else if (a.C == 64) launch_k(twell_transpose_kernel<64>, tgrid, TR_CHUNK, 0, sw, p);
    else launch_k(twell_transpose_kernel<128>, tgrid, TR_CHUNK, 0, sw, p);
    const cudaError_t r = cudaGetLastError();
    prof_mark(KID_BWD_TRANSPOSE, sw);
    return r;
  };
  auto dx_spmm = [&]() {
    if (bf) TW_VPT(bwd_dx_kernel, bf16, a.T, s, dx_passes, , dx_passes > 1);
    else TW_VPT(bwd_dx_kernel, float, a.T, s, dx_passes, , dx_passes > 1);
    const cudaError_t r = cudaGetLastError();
    prof_mark(KID_BWD_DX, s, dx_passes);
    return r;
  };
  // the transpose first when forked: it is short and heads the longer chain
  if (fork) {
    e = transpose();
    if (e == cudaSuccess) e = dx_spmm();
  } else {
    e = dx_spmm();
    if (e == cudaSuccess) e = transpose();
  }
  if (e == cudaSuccess) {  // 4. weight gradients
#define TW_PART0 , 0
#define TW_PART1 , 1
#define TW_PART2 , 2
    if (dw_split) {  // x rows (dW_gate, dW_up, dbg), then dy rows (dW_down)
      if (bf) {
        TW_VPT(bwd_dw_kernel, bf16, a.F, sw, dw_passes, TW_PART1, true);
        TW_VPT(bwd_dw_kernel, bf16, a.F, sw, dw_passes, TW_PART2, true);
      } else {
        TW_VPT(bwd_dw_kernel, float, a.F, sw, dw_passes, TW_PART1, true);
        TW_VPT(bwd_dw_kernel, float, a.F, sw, dw_passes, TW_PART2, true);
      }
    } else {
      if (bf) TW_VPT(bwd_dw_kernel, bf16, a.F, sw, dw_passes, TW_PART0, false);
      else TW_VPT(bwd_dw_kernel, float, a.F, sw, dw_passes, TW_PART0, false);
    }
#undef TW_PART0
#undef TW_PART1
#undef TW_PART2
    e = cudaGetLastError();
    prof_mark(KID_BWD_DW, sw, dw_passes * (dw_split ? 2 : 1));
  }
#undef TW_VPT
  // 5. weight gradients of the dense-path rows (added to those of step 4;
  // after the dense rows' dh on s3)
  if (e == cudaSuccess && gemm) {
    if (fork) e = cudaStreamWaitEvent(sw, aux->mid, 0);
    if (e == cudaSuccess) e = launch_tc_bwd_dw(a, sw);
    prof_mark(KID_BWD_DENSE_DW, sw);
  }
  if (fork) {  // join (also after an error, so the caller's stream stays ordered)
    const cudaError_t j1 = cudaEventRecord(aux->join, sw);
    const cudaError_t j2 = j1 == cudaSuccess ? cudaStreamWaitEvent(s, aux->join, 0) : j1;
    if (e == cudaSuccess) e = j2;
  }
  return join3(e);
}

}  // namespace twell

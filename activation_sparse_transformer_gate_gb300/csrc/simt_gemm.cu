// simt_gemm.cu -- CUDA-core (FFMA, fp32 accumulate, no TF32) tiled kernels:
//   * the gate matmul with the ReLU + TwELL packing epilogue, and
//   * the dense FFN rows of the hybrid fallback (gate+up, then down).
// These serve the fp32 configuration, whose tolerance rules out TF32 tensor
// cores; the bf16 configuration runs the tcgen05 kernels of tc_gemm.cu.
//
// "Sparser, Faster, Lighter Transformer Language Models", technical summary
// section 2.A: TwELL is materialised in the epilogue of the dense gate matmul;
// rows that overflow go to the dense backup and take the dense FFN.
#include "common.cuh"
#include "kernels.h"

namespace twell {

namespace {

constexpr int BM = 64, BK = 16, NT = 256;

// Load element (r, k) of a row-major [rows][ld] matrix as float, zero outside.
template <class T>
__device__ __forceinline__ float ld_el(const T *p, int r, int k, int rows, int cols, int ld) {
  return (r < rows && k < cols) ? to_f(p[(size_t)r * ld + k]) : 0.f;
}

}  // namespace

// ---------------------------------------------------------------------------
// Gate matmul + ReLU + TwELL pack.  CTA tile: 64 rows x BN (= C) columns, one
// TwELL tile per CTA column block.  Thread (ty, tx) owns rows ty + 16i and
// columns tx + 16j.  The epilogue stages z in shared memory and packs each
// row with one warp (ballot + popc ranks, ascending columns).
template <class T, int BN>
__global__ void __launch_bounds__(NT)
simt_gate_pack_kernel(const T *__restrict__ x, const T *__restrict__ Wg,
                      const float *__restrict__ bg, const float *__restrict__ rb, int Tn, int D,
                      int F, int K, uint8_t *__restrict__ idx, T *__restrict__ val,
                      uint8_t *__restrict__ nnz, uint32_t *__restrict__ ovf_bits,
                      T *__restrict__ wide, unsigned long long *__restrict__ slots) {
  pdl_begin();
  constexpr int TN = BN / 16;
  constexpr int E = BN / 32;
  __shared__ float smem[BM * (BN + 1) > BK * (BM + 4) + BK * (BN + 4) ? BM * (BN + 1)
                                                                      : BK * (BM + 4) + BK * (BN + 4)];
  float *As = smem;                 // [BK][BM+4]
  float *Bs = smem + BK * (BM + 4); // [BK][BN+4]
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const int m0 = blockIdx.y * BM, j = blockIdx.x, n0 = j * BN;
  float acc[4][TN];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int q = 0; q < TN; ++q) acc[i][q] = 0.f;

  for (int k0 = 0; k0 < D; k0 += BK) {
    // A tile: 64 x 16 = 4 per thread
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int e = tid + i * NT, r = e / BK, k = e % BK;
      As[k * (BM + 4) + r] = ld_el(x, m0 + r, k0 + k, Tn, D, D);
    }
    // B tile: BN x 16
#pragma unroll
    for (int i = 0; i < BN * BK / NT; ++i) {
      int e = tid + i * NT, r = e / BK, k = e % BK;
      Bs[k * (BN + 4) + r] = ld_el(Wg, n0 + r, k0 + k, F, D, D);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float a[4], b[TN];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k * (BM + 4) + ty + 16 * i];
#pragma unroll
      for (int q = 0; q < TN; ++q) b[q] = Bs[k * (BN + 4) + tx + 16 * q];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < TN; ++q) acc[i][q] = fmaf(a[i], b[q], acc[i][q]);
    }
    __syncthreads();
  }
  // z = acc + bg[n] + rb[t] staged as [BM][BN+1]
  float *Z = smem;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty + 16 * i;
    const float rbv = (rb && m0 + r < Tn) ? rb[m0 + r] : 0.f;
#pragma unroll
    for (int q = 0; q < TN; ++q) {
      const int c = tx + 16 * q;
      Z[r * (BN + 1) + c] = (acc[i][q] + bg[n0 + c]) + rbv;
    }
  }
  __syncthreads();
  const int lane = tid & 31, w = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  for (int r = w; r < BM; r += NT / 32) {
    const int t = m0 + r;
    if (t >= Tn) break;
    float v[E];
    unsigned m[E];
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      v[e] = Z[r * (BN + 1) + lane + 32 * e];
      m[e] = __ballot_sync(0xffffffffu, v[e] > 0.f);
      cnt += __popc(m[e]);
    }
    const size_t s0 = ((size_t)j * Tn + t) * (size_t)K;
    int before = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if ((m[e] >> lane) & 1u) {
        const int rk = before + __popc(m[e] & lt);
        if (rk < K) {
          idx[s0 + rk] = (uint8_t)(lane + 32 * e);
          val[s0 + rk] = from_f<T>(v[e]);
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
    if (lane == 0) {
      nnz[(size_t)j * Tn + t] = (uint8_t)cnt;
      if (cnt > K) atomicOr(&ovf_bits[t >> 5], 1u << (t & 31));
      if (filled && slots) atomicAdd(slots, (unsigned long long)filled);  // dispatcher's density
    }
    if (cnt > K) {  // overflowing (row, tile): keep the full ReLU(z) tile
      T *wd = wide + ((size_t)j * Tn + t) * BN;
#pragma unroll
      for (int e = 0; e < E; ++e) wd[lane + 32 * e] = from_f<T>(v[e] > 0.f ? v[e] : 0.f);
    }
  }
}

cudaError_t launch_simt_gate_pack(const FwdArgs &a, cudaStream_t s) {
  dim3 grid(a.F / a.C, (a.T + BM - 1) / BM);
#define TW_GP(TT, BNN)                                                                         \
  launch_k(simt_gate_pack_kernel<TT, BNN>, grid, NT, 0, s,                                     \
      (const TT *)a.x, (const TT *)a.Wg, a.bg, a.rb, a.T, a.D, a.F, a.K, a.tw.idx,             \
      (TT *)a.tw.val, a.tw.nnz, a.ws.ovf_bits, (TT *)a.ws.wide, &a.ws.ctl->slots)
  if (a.dtype == TWELL_BF16) {
    if (a.C == 32) TW_GP(bf16, 32); else if (a.C == 64) TW_GP(bf16, 64); else TW_GP(bf16, 128);
  } else {
    if (a.C == 32) TW_GP(float, 32); else if (a.C == 64) TW_GP(float, 64); else TW_GP(float, 128);
  }
#undef TW_GP
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Dense rows of the hybrid fallback.  Row m of the dense path is token
// tok(m) = m (all-dense mode) or rows[m] (hybrid mode); m < ctl->n_rows.
//  MODE_GU: z = x.Wg[n] + bg + rb, g = ReLU(z) rounded to T, u = x.Wu[n],
//           h = g*u (gated) or g -> h[m][n]; the overflow rows also get
//           g_fb[pos][n] (and u_fb[pos][n] when training).
//  MODE_D : y[tok][d] = sum_n h[m][n] Wd[n][d].
enum { MODE_GU = 0, MODE_D = 1 };

struct RowsParams {
  const void *x, *Wg, *Wu, *Wd;
  const float *bg, *rb;
  int Tn, D, F, cap, gated, train;
  const Ctl *ctl;
  const int32_t *rows, *pos;
  void *h, *g_fb, *u_fb, *y, *urows;
};

template <class T, int MODE>
__global__ void __launch_bounds__(NT) simt_rows_kernel(RowsParams p) {
  pdl_begin();
  constexpr int BN = 64;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[2][BK][BN + 4];
  const int n_rows = p.ctl->n_rows;
  const int dense = p.ctl->dense;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  if (m0 >= n_rows) return;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const int N = MODE == MODE_GU ? p.F : p.D;
  const int KD = MODE == MODE_GU ? p.D : p.F;
  const bool two = MODE == MODE_GU && p.gated;
  const T *A = MODE == MODE_GU ? (const T *)p.x : (const T *)p.h;
  float acc[2][4][4];
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[b][i][q] = 0.f;

  for (int k0 = 0; k0 < KD; k0 += BK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + i * NT, r = e / BK, k = e % BK;
      const int m = m0 + r;
      float v = 0.f;
      if (m < n_rows && k0 + k < KD) {
        const int src = MODE == MODE_GU ? (dense ? m : p.rows[m]) : m;
        v = to_f(A[(size_t)src * KD + k0 + k]);
      }
      As[k][r] = v;
    }
    if (MODE == MODE_GU) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = tid + i * NT, r = e / BK, k = e % BK;
        Bs[0][k][r] = ld_el((const T *)p.Wg, n0 + r, k0 + k, N, KD, KD);
        if (two) Bs[1][k][r] = ld_el((const T *)p.Wu, n0 + r, k0 + k, N, KD, KD);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = tid + i * NT, k = e / BN, c = e % BN;
        Bs[0][k][c] = ld_el((const T *)p.Wd, k0 + k, n0 + c, KD, N, N);
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        if (b == 1 && !two) break;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float bv = Bs[b][k][tx + 16 * q];
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[b][i][q] = fmaf(a[i], bv, acc[b][i][q]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= n_rows) continue;
    const int tok = dense ? m : p.rows[m];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + tx + 16 * q;
      if (n >= N) continue;
      if (MODE == MODE_GU) {
        float z = acc[0][i][q] + p.bg[n];
        if (p.rb) z += p.rb[tok];
        const float g = z > 0.f ? to_f(from_f<T>(z)) : 0.f;
        const float u = acc[1][i][q];
        const float hv = p.gated ? g * u : g;
        ((T *)p.h)[(size_t)m * p.F + n] = from_f<T>(hv);
        if (dense && p.train && p.gated) ((T *)p.urows)[(size_t)m * p.F + n] = from_f<T>(u);
        const int ps = dense ? p.pos[tok] : m;
        if (ps >= 0 && ps < p.cap) {
          ((T *)p.g_fb)[(size_t)ps * p.F + n] = from_f<T>(g);
          if (p.train && p.gated) ((T *)p.u_fb)[(size_t)ps * p.F + n] = from_f<T>(u);
        }
      } else {
        ((T *)p.y)[(size_t)tok * p.D + n] = from_f<T>(acc[0][i][q]);
      }
    }
  }
}

static RowsParams rows_params(const FwdArgs &a) {
  RowsParams p;
  p.x = a.x; p.Wg = a.Wg; p.Wu = a.Wu; p.Wd = a.Wd; p.bg = a.bg; p.rb = a.rb;
  p.Tn = a.T; p.D = a.D; p.F = a.F; p.cap = a.tw.ovf_cap; p.gated = a.gated; p.train = a.train;
  p.ctl = a.ws.ctl; p.rows = a.ws.rows; p.pos = a.ws.pos;
  p.h = a.ws.h; p.g_fb = a.tw.g_fb; p.u_fb = a.tw.u_fb; p.y = a.y; p.urows = a.ws.urows;
  return p;
}

cudaError_t launch_simt_dense_gu(const FwdArgs &a, cudaStream_t s) {
  RowsParams p = rows_params(a);
  dim3 g((a.F + 63) / 64, (a.T + BM - 1) / BM);
  if (a.dtype == TWELL_BF16) launch_k(simt_rows_kernel<bf16, MODE_GU>, g, NT, 0, s, p);
  else launch_k(simt_rows_kernel<float, MODE_GU>, g, NT, 0, s, p);
  return cudaGetLastError();
}

cudaError_t launch_simt_dense_down(const FwdArgs &a, cudaStream_t s) {
  RowsParams p = rows_params(a);
  dim3 g((a.D + 63) / 64, (a.T + BM - 1) / BM);
  if (a.dtype == TWELL_BF16) launch_k(simt_rows_kernel<bf16, MODE_D>, g, NT, 0, s, p);
  else launch_k(simt_rows_kernel<float, MODE_D>, g, NT, 0, s, p);
  return cudaGetLastError();
}

}  // namespace twell

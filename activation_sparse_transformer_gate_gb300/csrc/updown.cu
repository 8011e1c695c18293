// updown.cu -- fused sparse up + down projection over TwELL.
//
// "Sparser, Faster, Lighter Transformer Language Models", technical summary
// section 2.B (inference): one fused kernel performs the up and down
// projections in a single pass from the gate activations stored in TwELL,
// keeping global-memory traffic low and working from registers and shared
// memory.
//
// Design (GB300): one CTA of 4 warps per token.  The active pairs (neuron n,
// gate g) come from the token's TwELL slots, compacted into a shared-memory
// list.  Phase 1: each warp computes whole dot products u = x . W_up[n] for
// its share of the pairs (lane l owns the 16-byte vectors l, l+32, ... of the
// row; two rows in flight per warp; warp shuffles only), so no barrier sits
// inside the pair loop.  Phase 2: each thread owns a d_model slice of y (two
// 16-byte vectors at d_model 2048, which halves the per-row address and loop
// work of one) and accumulates h * W_down[n] over all pairs with 128-bit
// coalesced row loads, 8 rows in flight.  One barrier per tile group separates
// the phases.  All-dense mode (and overflow rows when there are many) is left
// to the tensor-core dense-row GEMMs; a few overflow rows are handled here
// from the wide-tile buffer.
//
// Two passes when W_up and W_down together do not fit in L2: with both in
// one pass every token's CTA reads rows of both, the working set is both
// matrices, and rows miss L2 (d_model 4096 / d_ff 14336 bf16, 235 MB: 47% L2
// hits, 5.4 GB of DRAM reads for 9.4 GB gathered; random-row gathers of the
// two matrices in that order run at 11.0 TB/s on GB300, one matrix at a time
// at 15.7 TB/s).  The up pass then computes h = g u of every slot into an
// fp32 slot array (the same values the fused kernel keeps in shared memory),
// and the down pass reads them back: each pass's working set is one matrix.
// Overflow rows handled here run both phases in the up pass.
#include "common.cuh"
#include "gather.cuh"
#include "kernels.h"

namespace twell {

namespace {

constexpr int UD_THREADS = 128;  // 4 warps per token CTA
// Rows of W_down in flight per batch of the down phase, exact row shapes:
// 24 / VPT vectors per thread (12 rows at d_model 2048 bf16), but 4 rows
// at VPT 4 and 1 at VPT 8, where more spill registers: at d_model 4096 the
// 6-row batch spilled and 4 rows took the kernel from 0.93 to 0.74 ms
// (8192 tokens, d_ff 14336, 0.49% active).  At d_model 2048, 8 or 6 rows
// with five CTAs per SM were slower than 12 with four (0.194 -> 0.211 /
// 0.222 ms at 4096 tokens, d_ff 8192).
template <int VPT>
constexpr int exact_rows() { return VPT == 4 ? 4 : VPT == 8 ? 1 : 24 / VPT; }
// Rows in flight for the other shapes (predicated loads): 16 / VPT, one at
// VPT 8 (d_model 8192 bf16), where two spill.
template <int VPT>
constexpr int generic_rows() { return VPT == 8 ? 1 : 16 / VPT; }

struct UDParams {
  const void *x, *Wu, *Wd;
  const uint8_t *idx, *nnz;
  const void *val, *wide;
  void *u_val, *y, *g_fb, *u_fb;
  const int32_t *pos;
  float *hsl;   // [F/C][T][K] h at the slots between the two passes
  int Tn, D, F, C, K, gated, train, cap;
  int phase;    // 0: up and down in one pass; 1: up pass; 2: down pass
  const Ctl *ctl;
  int32_t *status;
};

}  // namespace

// One CTA (4 warps) per token.  Rows that run on the dense GEMM path
// (all-dense mode, or overflow rows when there are many) are skipped; an
// overflow row handled here takes its overflowing tiles from the wide-tile
// buffer and also writes its dense backup row (g_fb, and u_fb when training).
// Per tile group: phase 1 -- warp w computes the full dot products
// u = x . W_up[n] of pairs w, w+4, ... (two rows in flight per warp, warp
// shuffles only); one barrier; phase 2 -- every thread accumulates its slice
// of y += h * W_down[n] over all pairs, 8 rows in flight, no barrier.
template <class T, int VPT, int VPL, int PIF, int PB2, bool EXACT>
__global__ void __launch_bounds__(UD_THREADS, 4) updown_fused_kernel(UDParams p) {
  pdl_begin();
  constexpr int EV = Vec<T>::EV;
  __shared__ int s_n[LIST_CAP];
  __shared__ float s_g[LIST_CAP];
  __shared__ int s_slot[LIST_CAP];
  __shared__ uint4 s_x[1024];  // x_t, read by every warp in phase 1
  __shared__ int s_wsum[32];
  __shared__ int s_total;

  if (p.ctl->dense) return;
  const int t = blockIdx.x;
  const int ps = p.pos[t];
  const bool ovf = ps >= 0;
  if (ovf && p.ctl->ovf_gemm) return;
  if (ovf && p.phase == 2) return;               // done in the up pass
  const bool up_only = p.phase == 1 && !ovf;     // h to the slot array, no y
  const bool down_only = p.phase == 2;           // h from the slot array
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
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
  if (p.gated && !down_only)  // x_t to shared memory (visible after the barriers of build_pairs)
    for (int v = tid; v < NV; v += blockDim.x)  // x_t is read once here: evict-first
      s_x[v] = ldg_stream<L2_FIRST>((const uint4 *)p.x + (size_t)t * NV + v);
  float2 yr[VPT][EV / 2];
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int e = 0; e < EV / 2; ++e) yr[v][e] = make_float2(0.f, 0.f);
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
    // ---- phase 1: u and h of every pair, one warp per pair ------------------
    if (p.gated && !down_only && VPL > 16) {
      // rows of more than 16 vectors per lane (d_model 8192 bf16): one row
      // per warp, loaded and dotted 16 vectors per lane at a time (the whole
      // row in registers would spill); the partial sums run in one order
      for (int i = w; i < P; i += nw) {
        const uint4 *row = Wu4 + (size_t)s_n[i] * NV;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll 1
        for (int h = 0; h < VPL; h += 16) {
          uint4 wr[16];
          warp_row<16, L2_NORMAL, EXACT>(row + 32 * h, NV - 32 * h, true, wr);
          warp_dot_smem_acc<T, 16>(s_x + 32 * h, NV - 32 * h, wr, s0, s1);
        }
        float u = s0 + s1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
        if (lane == 0) {
          s_g[i] *= u;  // h = g * u, in place
          if (p.train) {
            const int sl = s_slot[i];
            if (sl >= 0) ((T *)p.u_val)[sl] = from_f<T>(u);
            else if (fb && sl != PAD_SLOT) ((T *)p.u_fb)[(size_t)ps * p.F + (-1 - sl)] = from_f<T>(u);
          }
        }
      }
    } else if (p.gated && !down_only) {
      for (int i0 = w; i0 < P; i0 += nw * PIF) {
        uint4 wr[PIF][VPL];
#pragma unroll
        for (int q = 0; q < PIF; ++q) {
          const int i = i0 + q * nw;
          // exact rows: load the (valid, clamped) row unconditionally, discard its dot
          warp_row<VPL, L2_NORMAL, EXACT>(Wu4 + (size_t)s_n[i < P ? i : i0] * NV, NV, EXACT || i < P, wr[q]);
        }
        // x_t: with one row in flight per warp it is read from shared memory
        // vector by vector inside the dot (no registers held for it across
        // the row loads); with two, once into registers for both rows
        constexpr bool XS = PIF == 1;
        uint4 xw[XS ? 1 : VPL];
        if (!XS) {
#pragma unroll
          for (int k = 0; k < VPL; ++k) {
            const int vi = lane + 32 * k;
            xw[k] = (EXACT || vi < NV) ? s_x[vi] : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int q = 0; q < PIF; ++q) {
          const int i = i0 + q * nw;
          float u;
          if constexpr (XS) u = warp_dot_smem<T, VPL>(s_x, NV, wr[q]);
          else u = warp_dot<T, VPL>(reinterpret_cast<const uint4(&)[VPL]>(xw), wr[q]);
          if (lane == 0 && i < P) {
            s_g[i] *= u;  // h = g * u, in place
            if (p.train) {
              const int sl = s_slot[i];
              if (sl >= 0) ((T *)p.u_val)[sl] = from_f<T>(u);
              else if (fb && sl != PAD_SLOT) ((T *)p.u_fb)[(size_t)ps * p.F + (-1 - sl)] = from_f<T>(u);
            }
          }
        }
      }
    }
    if (down_only)  // h of the up pass (slots of a non-overflow row are >= 0)
      for (int i = tid; i < P; i += blockDim.x) s_g[i] = p.hsl[s_slot[i]];
    __syncthreads();
    if (up_only) {
      for (int i = tid; i < P; i += blockDim.x) p.hsl[s_slot[i]] = s_g[i];
      __syncthreads();  // the list is rewritten by the next group
      continue;
    }
    // ---- phase 2: y += h * W_down[n], thread-owned slices -------------------
    for (int b0 = 0; b0 < P; b0 += PB2) {
      const int nb = P - b0 < PB2 ? P - b0 : PB2;
      uint4 wd[PB2][VPT];
      if (EXACT && nb == PB2) gather8<T, VPT, PB2, UD_THREADS>(Wd4, s_n, b0, nb, NV, NV, wd);
      else gather8<T, VPT, PB2>(Wd4, s_n, b0, nb, NV, NV, wd);
#pragma unroll
      for (int b = 0; b < PB2; ++b) {
        if (b >= nb) break;
        const float h = s_g[b0 + b];
#pragma unroll
        for (int v = 0; v < VPT; ++v) axpy_vec<T>(yr[v], h, wd[b][v]);
      }
    }
    __syncthreads();  // the list is rewritten by the next group
  }

  if (up_only) return;
  uint4 *yrow = (uint4 *)p.y + (size_t)t * NV;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int vi = tid + v * blockDim.x;
    if (vi < NV) stg_stream(yrow + vi, Vec<T>::pack(reinterpret_cast<const float *>(yr[v])));
  }
}

cudaError_t launch_updown_fused(const FwdArgs &a, cudaStream_t s, int *launches) {
  UDParams p;
  p.x = a.x; p.Wu = a.Wu; p.Wd = a.Wd; p.idx = a.tw.idx; p.nnz = a.tw.nnz; p.val = a.tw.val;
  p.wide = a.ws.wide; p.u_val = a.tw.u_val; p.y = a.y; p.g_fb = a.tw.g_fb; p.u_fb = a.tw.u_fb;
  p.pos = a.ws.pos; p.Tn = a.T; p.D = a.D; p.F = a.F; p.C = a.C; p.K = a.K; p.gated = a.gated;
  p.train = a.train && a.gated; p.cap = a.tw.ovf_cap; p.ctl = a.ws.ctl; p.status = a.tw.status;
  p.hsl = a.ws.hs;
  // one pass, or the up pass then the down pass (gated FFN whose two
  // gathered matrices do not fit in L2 together)
  const size_t es = a.dtype == TWELL_BF16 ? 2 : 4;
  const bool two = a.gated && gather_passes(a.tw.gather_passes, 2.0 * a.F * a.D * es, a.D * es / 16, 1) > 1;
  if (launches) *launches = two ? 2 : 1;
  const int EV = a.dtype == TWELL_BF16 ? 8 : 4;
  const int NV = a.D / EV;  // <= 1024 (checked by the caller)
  const int vpl = NV <= 32 ? 1 : NV <= 64 ? 2 : NV <= 128 ? 4 : NV <= 256 ? 8 : NV <= 512 ? 16 : 32;
#define TW_UD(TT, L)                                                                           \
  do {                                                                                         \
    constexpr int VPT_ = (L + 3) / 4;                                                          \
    for (int ph = two ? 1 : 0; ph <= (two ? 2 : 0); ++ph) {                                    \
      p.phase = ph;                                                                            \
      if (NV == 32 * (L) && NV == VPT_ * UD_THREADS)                                           \
        launch_k(updown_fused_kernel<TT, VPT_, L, (L <= 8 ? 2 : 1), exact_rows<VPT_>(), true>, a.T,  \
                 UD_THREADS, 0, s, p);                                                         \
      else                                                                                     \
        launch_k(updown_fused_kernel<TT, VPT_, L, (L <= 8 ? 2 : 1), generic_rows<VPT_>(), false>, a.T, \
                 UD_THREADS, 0, s, p);                                                         \
    }                                                                                          \
  } while (0)
#define TW_UD_T(TT)                                                                            \
  do {                                                                                         \
    switch (vpl) {                                                                             \
      case 1: TW_UD(TT, 1); break;                                                             \
      case 2: TW_UD(TT, 2); break;                                                             \
      case 4: TW_UD(TT, 4); break;                                                             \
      case 8: TW_UD(TT, 8); break;                                                             \
      case 16: TW_UD(TT, 16); break;                                                           \
      default: TW_UD(TT, 32); break;                                                           \
    }                                                                                          \
  } while (0)
  if (a.dtype == TWELL_BF16) TW_UD_T(bf16);
  else TW_UD_T(float);
#undef TW_UD_T
#undef TW_UD
  return cudaGetLastError();
}

}  // namespace twell

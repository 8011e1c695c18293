// tc_gemm.cu -- tcgen05 (5th-generation tensor core) GEMM engine for the bf16
// path, with the epilogues of the TwELL FFN:
//   EPI_PACK : z = x Wg^T + bg + rb -> ReLU -> TwELL slots + nnz     (gate)
//   EPI_GU   : g = ReLU(z) rounded to bf16 (B = Wg; with a second B = Wu
//              also u and h = g*u) -> h rows (+ g_fb / u_fb rows of overflow
//              rows); the plain FFN's dense rows                (dense rows)
//   EPI_DOWN : y[tok] = h Wd, Wd read MN-major straight from [F][D]   (dense rows)
//              (gated FFN: h and a copy of Wd in fp16, see below)
//   EPI_U    : the gated FFN's dense rows: B = Wu only, g read back from the
//              TwELL slots / wide tiles, h = g*u (+ u at the slots)   (dense rows)
//   EPI_DH   : dh = dy Wd^T + lambda sign(h) -> dz, du, h rows (fp16) and
//              column sums of dz                                  (bwd rows)
//   EPI_DHS  : the same dh for the rows left to the gathers, read only at the
//              TwELL slots (and the overflow rows' backup-row columns) ->
//              fp32 dz, du, h where the gather SDDMM puts them   (bwd, sparse)
//   EPI_DX   : dx[tok] = dz Wg + du Wu (two K ranges, B MN-major) (bwd rows)
//   EPI_DW   : dW = A^T B with A, B both MN-major (token axis = K), fp32
//              rows stored or added                               (bwd rows)
//
// Precision of the dense-path rows.  Their activations h = g u and their
// gradients dz, du, h are formed in fp32 and enter the tensor cores as MMA
// operands.  One bf16 rounding of them would give output errors of 1-5% of
// rms at the largest elements (where a few large activations dominate a
// row), so these GEMMs take fp16 operands (kind::f16 with F16 A and B): 2^-11
// relative rounding, about an eighth of that error, at the cost of one GEMM.
// The other operand (W_down, W_gate, W_up, x, dy: bf16) is copied to fp16,
// which is exact for values of magnitude within [2^-14, 65504]; larger ones
// would not be representable (TWELL_ERR_RANGE).
//   EPI_F32  : plain fp32 C = A B^T, A B or A^T B (test hook)
//
// "Sparser, Faster, Lighter Transformer Language Models", technical summary
// section 2.A: TwELL is materialised in the epilogue of an optimised dense
// matmul, with no synchronisation between CTAs; each CTA owns whole tiles.
//
// Structure (one CTA per SM, persistent over output tiles, 192 threads):
//   warp 0      TMA producer: A and B tiles (128B-swizzled) into a ring of
//               shared-memory stages, completion counted on mbarriers.
//   warp 1      allocates TMEM; one elected lane issues tcgen05.mma
//               (M=128, N=BN, K=16, bf16 in, fp32 accumulate in TMEM) and
//               commits each stage back to the producer and each finished
//               accumulator to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld 32x32b (thread = accumulator row),
//               fused element-wise work and stores.  Two TMEM accumulators
//               alternate so the epilogue of tile i overlaps the MMAs of i+1.
// Every mbarrier wait of the pipeline is bounded by a global-timer limit
// (TWELL_WAIT_LIMIT_NS, 2 s unless the build sets another); on expiry the CTA
// records TWELL_ERR_TIMEOUT in the status word, waits (with a fixed 2 s limit
// of its own) for the copies and MMAs it has in flight, frees its TMEM and
// returns.  The four epilogue warps take the outcome of each wait together,
// so they leave their loop at the same tile.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "test_hooks.h"

namespace twell {

namespace {

constexpr int BM = 128, BK = 64, NTHREADS = 192;
// bf16 elements per row of the EPI_U g staging: 32 columns, a spare element
// for scattered slots outside the block, padding to 16 bytes
constexpr int GZ_STRIDE = 40;
// Limit of a pipeline wait (a build may shorten it to make the waits run out
// on a sane input: the timeout path is then exercised without a fault).
#ifndef TWELL_WAIT_LIMIT_NS
#define TWELL_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr uint64_t WAIT_LIMIT_NS = TWELL_WAIT_LIMIT_NS;
// Limit of the waits for work already in flight before a CTA exits (TMA
// copies into shared memory, MMAs writing TMEM): always long, since leaving
// earlier would free memory that the hardware still writes.
constexpr uint64_t DRAIN_LIMIT_NS = 2000000000ull;

enum Epi { EPI_PACK = 0, EPI_GU = 1, EPI_DOWN = 2, EPI_F32 = 3, EPI_U = 4, EPI_DH = 5, EPI_DX = 6,
           EPI_DW = 7, EPI_DHS = 8 };
// fp32 elements per row of the EPI_DHS accumulator staging (32 columns; the
// 144-byte stride keeps the 16-byte stores of 8 consecutive rows on
// distinct banks)
constexpr int DHS_STRIDE = 36;

// ---------------------------------------------------------------- PTX ----
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait.  Returns false (and raises the CTA-wide abort flag and the
// device status) when the limit expires or another role has aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer() - t0 > WAIT_LIMIT_NS) {
      *abort_flag = 1;
      set_status(status, TWELL_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a 128B-swizzled operand tile.
//  [0,14) start>>4  [16,30) LBO>>4  [32,46) SBO>>4  [46,48) version 1
//  [61,64) layout 2 = SWIZZLE_128B
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D=f32 (bits 4-5), A and B both bf16
// (bits 7-9 and 10-12 = 1) or both fp16 (= 0), A and B each K- or MN-major
// (bits 15 and 16), N>>3 at bit 17, M>>4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool a_mn, bool b_mn, bool f16) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane.  The
// wait is inside the same asm statement, so no use of the outputs can be
// scheduled before the load has completed.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The K slots of one (row, tile) with vector loads (K in {1,2,4,8,16,32}; a
// slot row starts at a multiple of its own size, so each load is aligned):
// load_idx gives the idx bytes, load_vals the bf16 value pairs; words past
// the slots are zero.
__device__ __forceinline__ void load_idx(const uint8_t *ip, int K, uint32_t (&iw)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) iw[i] = 0u;
  if (K >= 16) {
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (q * 16 < K) {
        const uint4 a = ((const uint4 *)ip)[q];
        iw[4 * q] = a.x; iw[4 * q + 1] = a.y; iw[4 * q + 2] = a.z; iw[4 * q + 3] = a.w;
      }
  } else if (K == 8) {
    const uint2 a = *(const uint2 *)ip;
    iw[0] = a.x; iw[1] = a.y;
  } else if (K == 4) {
    iw[0] = *(const uint32_t *)ip;
  } else if (K == 2) {
    iw[0] = *(const uint16_t *)ip;
  } else {
    iw[0] = *ip;
  }
}

__device__ __forceinline__ void load_vals(const bf16 *vp, int K, uint32_t (&vw)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) vw[i] = 0u;
  if (K >= 8) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q * 8 < K) {
        const uint4 a = ((const uint4 *)vp)[q];
        vw[4 * q] = a.x; vw[4 * q + 1] = a.y; vw[4 * q + 2] = a.z; vw[4 * q + 3] = a.w;
      }
  } else if (K == 4) {
    const uint2 a = *(const uint2 *)vp;
    vw[0] = a.x; vw[1] = a.y;
  } else if (K == 2) {
    vw[0] = *(const uint32_t *)vp;
  } else {
    vw[0] = *(const uint16_t *)vp;
  }
}

__device__ __forceinline__ void load_slots(const uint8_t *ip, const bf16 *vp, int K,
                                           uint32_t (&iw)[8], uint32_t (&vw)[16]) {
  load_idx(ip, K, iw);
  load_vals(vp, K, vw);
}

// Slot k's local column and bf16 value bits from the words of load_slots.
__device__ __forceinline__ int slot_col(const uint32_t (&iw)[8], int k) {
  return (int)((iw[k >> 2] >> (8 * (k & 3))) & 0xFFu);
}
__device__ __forceinline__ unsigned short slot_val(const uint32_t (&vw)[16], int k) {
  return (unsigned short)(vw[k >> 1] >> (16 * (k & 1)));
}

// 32 fp32 values as fp16 (round to nearest even), 64 bytes; a value beyond
// the fp16 range records TWELL_ERR_RANGE.
__device__ __forceinline__ void store_f16x32(__half *dst, const float (&v)[32], int32_t *status) {
  uint32_t w[16];
  bool big = false;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    big |= fabsf(v[i]) > 65504.f || fabsf(v[i + 1]) > 65504.f;
    __half2 h = __floats2half2_rn(v[i], v[i + 1]);
    w[i / 2] = *reinterpret_cast<uint32_t *>(&h);
  }
  if (big) set_status(status, TWELL_ERR_RANGE);
  uint4 *d4 = (uint4 *)dst;
#pragma unroll
  for (int v4 = 0; v4 < 4; ++v4)
    d4[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
}

__device__ __forceinline__ void epi_bar() {  // named barrier of the 4 epilogue warps
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// The same barrier with an AND of v over the 128 epilogue threads: every
// thread gets the same answer, so a decision taken on it is uniform (the
// warp-collective tcgen05.ld and the named barrier need all four warps on
// the same path).
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 128, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// --------------------------------------------------------------- params --
// Operand tensor maps.  a[0] / b[0]: gathered rows (dense-path rows of the
// hybrid), a[1] / b[1]: the operand in place (all-dense mode), or the second
// operand (EPI_GU: W_up; EPI_DX: du and W_up).  EPI_DW: A of problem q is
// a[q]; B is b[0] / b[1] (x), or b[2] / b[3] (dy) for the last problem.
struct TcMaps {
  CUtensorMap a[3];
  CUtensorMap b[4];
};

struct TcParams {
  int M_host;              // rows when m_dev == nullptr
  const int32_t *m_dev;    // device row count (dense path: ctl->n_rows)
  const int32_t *k_dev;    // device contraction length (EPI_DW: ctl->n_rows), else Kdim
  const Ctl *ctl;          // dense-path control (EPI_GU / EPI_DOWN), else null
  int N, Kdim;             // output columns, contraction length
  int Tn, F, D, C, Kslots, cap, gated, train;
  int Tp;                  // rows of the dense-path row buffers
  long long l2_bytes;      // L2 size of the device (tile order)
  const float *bg, *rb;
  const int32_t *rows, *pos;
  uint8_t *idx, *nnz;
  uint32_t *ovf_bits;
  unsigned long long *slots;  // EPI_PACK: total slots written (the dispatcher's density)
  bf16 *val, *uval;         // uval: u at the slots (backward)
  bf16 *h, *g_fb, *u_fb, *y;
  bf16 *wide;
  float *out;              // EPI_F32, EPI_DW
  float lambda;            // EPI_DH: L1 coefficient
  __half *dz2, *du2, *h2;  // EPI_DH outputs, [Tp][F] fp16
  float *dbg_r;            // EPI_DH: column sums of dz per 32-row group [group][F]; EPI_DW:
                           // summed over the groups in order and added to dbg_out
  float *dbg_out;          // EPI_DW: dbg (added from dbg_r with the W_gate problem)
  float *outq[3];          // EPI_DW: the fp32 output of each problem (dWg, [dWu,] dWd)
  int nq;                  // EPI_DW: problems in the launch
  float *sdz, *sdu, *shs;  // EPI_DHS: dz, du, h at the slots, [F/C][T][K]
  float *rdz, *rdu, *rhs;  // EPI_DHS: the same for overflow rows, [cap][F]
  int32_t *col_chunk;      // EPI_DHS: the sparse transpose's column counts
  int32_t *status;
};

// (M-block, N-block) of tile t: groups of gm M-blocks (the last one may be
// smaller), N-blocks outer and M-blocks inner within a group.
__device__ __forceinline__ void tile_mn(int t, int m_blocks, int n_blocks, int gm, int &mb,
                                        int &nb) {
  const int g = t / (gm * n_blocks);
  const int m0 = g * gm;
  const int gs = min(gm, m_blocks - m0);
  const int r = t - g * gm * n_blocks;
  nb = r / gs;
  mb = m0 + r % gs;
}

// nnz and the K slots (idx bytes, bf16 value pairs) of the TwELL tile that
// holds column col of row tok; the slot words are read even when the tile
// overflowed (then unused), so no load waits on another.
__device__ __forceinline__ void fetch_slots(const TcParams &p, int col, int tok, int &nz,
                                            uint32_t (&iw)[8], uint32_t (&vw)[16]) {
  const size_t jt = (size_t)(col / p.C) * p.Tn + tok;
  nz = p.nnz[jt];
  load_slots(p.idx + jt * p.Kslots, p.val + jt * p.Kslots, p.Kslots, iw, vw);
}

// EPI_DHS with two 128-column TwELL tiles per output tile and K <= 8: what
// one row needs of both tiles (its dense-backup position, and per tile the
// count, the slot indices, g and u at the slots), in compact registers.
struct DhsSlots {
  int ps, nz0, nz1;
  uint32_t i0[2], v0[4], q0[4], i1[2], v1[4], q1[4];
};

__device__ __forceinline__ void dhs_fetch(const TcParams &p, int tok, bool row_ok, int n0,
                                          DhsSlots &S) {
  S.ps = row_ok ? p.pos[tok] : -1;
  S.nz0 = S.nz1 = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) S.i0[i] = S.i1[i] = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) S.v0[i] = S.q0[i] = S.v1[i] = S.q1[i] = 0u;
  if (!row_ok || S.ps >= 0) return;
  uint32_t iw[8], vw[16];
  const size_t j0 = (size_t)(n0 / 128) * p.Tn + tok;
  S.nz0 = p.nnz[j0];
  load_idx(p.idx + j0 * p.Kslots, p.Kslots, iw);
  S.i0[0] = iw[0]; S.i0[1] = iw[1];
  load_vals(p.val + j0 * p.Kslots, p.Kslots, vw);
#pragma unroll
  for (int i = 0; i < 4; ++i) S.v0[i] = vw[i];
  if (p.gated) {
    load_vals(p.uval + j0 * p.Kslots, p.Kslots, vw);
#pragma unroll
    for (int i = 0; i < 4; ++i) S.q0[i] = vw[i];
  }
  if (n0 + 128 >= p.N) return;
  const size_t j1 = j0 + p.Tn;
  S.nz1 = p.nnz[j1];
  load_idx(p.idx + j1 * p.Kslots, p.Kslots, iw);
  S.i1[0] = iw[0]; S.i1[1] = iw[1];
  load_vals(p.val + j1 * p.Kslots, p.Kslots, vw);
#pragma unroll
  for (int i = 0; i < 4; ++i) S.v1[i] = vw[i];
  if (p.gated) {
    load_vals(p.uval + j1 * p.Kslots, p.Kslots, vw);
#pragma unroll
    for (int i = 0; i < 4; ++i) S.q1[i] = vw[i];
  }
}

// EPI_DHS: the gradients of one TwELL tile's slots (tile j, row tok) from dh
// at the slots, as the gather SDDMM finishes an entry: h = g u, dh += lambda
// sign(h), dz = [g > 0] dh u, du = [g > 0] dh g (plain FFN: u = 1), stored
// at the live slots (groups of four from the first; pad slots past the last
// group are not written, as no reader goes past nnz) with the sparse
// transpose's count of each live slot's column.  iw / vw / qw: the slot
// words of load_slots and of u at the slots; NK slots at most (K <= NK).
template <int NK>
__device__ __forceinline__ void dhs_store_slots(const TcParams &p, int j, int tok, int K, int nz,
                                                const uint32_t (&iw)[NK / 4 > 0 ? NK / 4 : 1],
                                                const uint32_t (&vw)[NK / 2],
                                                const uint32_t (&qw)[NK / 2],
                                                const float (&dh)[NK], int nch) {
  const size_t s0 = ((size_t)j * p.Tn + tok) * K;
#pragma unroll
  for (int k0 = 0; k0 < NK; k0 += 4) {
    if (k0 >= K) break;   // uniform
    if (k0 >= nz) break;  // no live slot left
    float dz[4], du[4], hv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = k0 + i;
      const bool live = k < nz;  // (pad slots store zeros)
      const uint32_t gb = (vw[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
      const uint32_t ub = (qw[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
      const float g = live ? __uint_as_float(gb << 16) : 0.f;
      const float u = !p.gated ? 1.f : (live ? __uint_as_float(ub << 16) : 0.f);
      const float h = p.gated ? g * u : g;
      const float d = dh[k] + p.lambda * (h > 0.f ? 1.f : (h < 0.f ? -1.f : 0.f));
      const bool act = g > 0.f;
      dz[i] = act ? (p.gated ? d * u : d) : 0.f;
      du[i] = act ? d * g : 0.f;
      hv[i] = h;
      const int c = (int)((iw[k >> 2] >> (8 * (k & 3))) & 0xFFu);
      if (live && c < p.C)  // the transpose's count (a malformed index is not listed)
        atomicAdd(&p.col_chunk[((size_t)j * nch + tok / TR_CHUNK) * p.C + c], 1);
      else if (live)
        set_status(p.status, TWELL_ERR_INDEX);
    }
    if (K % 4 == 0) {
      *(float4 *)(p.sdz + s0 + k0) = make_float4(dz[0], dz[1], dz[2], dz[3]);
      *(float4 *)(p.sdu + s0 + k0) = make_float4(du[0], du[1], du[2], du[3]);
      *(float4 *)(p.shs + s0 + k0) = make_float4(hv[0], hv[1], hv[2], hv[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (k0 + i >= K) break;
        p.sdz[s0 + k0 + i] = dz[i];
        p.sdu[s0 + k0 + i] = du[i];
        p.shs[s0 + k0 + i] = hv[i];
      }
    }
  }
}

// EPI_DHS, an overflow row with a dense backup row (position ps): dz, du, h
// of the 32 columns from column col on, written in full to the overflow-row
// arrays (zeros where g = 0).
__device__ __forceinline__ void dhs_store_row_block(const TcParams &p, int ps, int col,
                                                    const float (&v)[32]) {
  const size_t o = (size_t)ps * p.F + col;
  const uint4 *gr = (const uint4 *)(p.g_fb + o);
  const uint4 *ur = (const uint4 *)(p.u_fb + o);
  float4 *dz4 = (float4 *)(p.rdz + o), *du4 = (float4 *)(p.rdu + o), *h4 = (float4 *)(p.rhs + o);
#pragma unroll
  for (int v4 = 0; v4 < 4; ++v4) {
    const uint4 gv = gr[v4];
    const uint4 uv = p.gated ? ur[v4] : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u,
                                                   0x3F803F80u);  // u = 1
    const uint32_t ga[4] = {gv.x, gv.y, gv.z, gv.w}, ua[4] = {uv.x, uv.y, uv.z, uv.w};
    float dz[8], du[8], hv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float g = (e & 1) ? bf_hi(ga[e / 2]) : bf_lo(ga[e / 2]);
      const float u = (e & 1) ? bf_hi(ua[e / 2]) : bf_lo(ua[e / 2]);
      const float h = p.gated ? g * u : g;
      const float dh = v[8 * v4 + e] + p.lambda * (h > 0.f ? 1.f : (h < 0.f ? -1.f : 0.f));
      const bool act = g > 0.f;
      dz[e] = act ? (p.gated ? dh * u : dh) : 0.f;
      du[e] = act ? dh * g : 0.f;
      hv[e] = h;
    }
    dz4[2 * v4] = make_float4(dz[0], dz[1], dz[2], dz[3]);
    dz4[2 * v4 + 1] = make_float4(dz[4], dz[5], dz[6], dz[7]);
    du4[2 * v4] = make_float4(du[0], du[1], du[2], du[3]);
    du4[2 * v4 + 1] = make_float4(du[4], du[5], du[6], du[7]);
    h4[2 * v4] = make_float4(hv[0], hv[1], hv[2], hv[3]);
    h4[2 * v4 + 1] = make_float4(hv[4], hv[5], hv[6], hv[7]);
  }
}

// EPI_DHS: copy the accumulator block v into the thread's shared-memory row
// st, then dh[k] = the value at slot k's column for the slots in the block
// (local columns cl .. cl + 31 of the TwELL tile).
template <int NK>
__device__ __forceinline__ void dhs_pick(float *st, const float (&v)[32], int cl, int K, int nz,
                                         const uint32_t (&iw)[NK / 4 > 0 ? NK / 4 : 1],
                                         float (&dh)[NK]) {
  float4 *s4 = (float4 *)st;
#pragma unroll
  for (int v4 = 0; v4 < 8; ++v4)
    s4[v4] = make_float4(v[4 * v4], v[4 * v4 + 1], v[4 * v4 + 2], v[4 * v4 + 3]);
#pragma unroll
  for (int k = 0; k < NK; ++k) {
    if (k >= K) break;  // uniform
    const int c = (int)((iw[k >> 2] >> (8 * (k & 3))) & 0xFFu) - cl;
    if (k < nz && (unsigned)c < 32u) dh[k] = st[c];
  }
}

// The 32-column blocks of a TwELL tile (C columns) that hold one of the
// first nz slots.  A malformed index (>= C) names no block: it would
// otherwise set a bit of a block past the tile (the next tile's, where two
// tiles share an output tile).
template <int NK>
__device__ __forceinline__ uint32_t dhs_blocks(const uint32_t (&iw)[NK / 4 > 0 ? NK / 4 : 1],
                                               int K, int nz, int C) {
  uint32_t blk = 0;
#pragma unroll
  for (int k = 0; k < NK; ++k) {
    if (k >= K) break;  // uniform
    const int c = (int)((iw[k >> 2] >> (8 * (k & 3))) & 0xFFu);
    if (k < nz && c < C) blk |= 1u << (c >> 5);
  }
  return blk;
}

template <int BN, int NB, bool B_MN, int EPI, bool A_MN = false>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + NB * B_BYTES;
  static constexpr int STAGES = (200 * 1024) / STAGE_BYTES;
  static constexpr int TMEM_COLS_USED = 2 * NB * BN;
  static constexpr int TMEM_COLS = TMEM_COLS_USED <= 32 ? 32 : TMEM_COLS_USED <= 64 ? 64
                                   : TMEM_COLS_USED <= 128 ? 128 : TMEM_COLS_USED <= 256 ? 256
                                                                                         : 512;
  // EPI_PACK: per row idx (32 B) + bf16 val (64 B) slots, K <= 32, and a
  // 32-column bf16 staging row (64 B)
  static constexpr int SLOT_BYTES = EPI == EPI_PACK ? 128 * 32 * 3 + 128 * 64
                                    : EPI == EPI_U  ? 128 * GZ_STRIDE * 2 + 128 * 64  // g and u rows
                                    : EPI == EPI_DH ? 128 * GZ_STRIDE * 4  // g and u rows
                                    : EPI == EPI_DHS ? 128 * DHS_STRIDE * 4  // accumulator rows
                                                    : 0;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 256 + BN * 4 + SLOT_BYTES;
  static_assert(STAGES >= 2, "too few stages");
  static_assert(TMEM_COLS_USED <= 512, "TMEM overflow");
};

}  // namespace

template <int BN, int NB, bool B_MN, int EPI, bool A_MN = false, bool F16 = false>
__global__ void __launch_bounds__(NTHREADS, 1)
tc_gemm_kernel(const __grid_constant__ TcMaps maps, TcParams p) {
  pdl_begin();
  using CF = Cfg<BN, NB, B_MN, EPI, A_MN>;
  constexpr int S = CF::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *stages = smem;
  // full[S] empty[S] tfull[2] tempty[2] mma_done
  uint64_t *bars = (uint64_t *)(smem + S * CF::STAGE_BYTES);
  uint32_t *tmem_slot = (uint32_t *)(bars + 2 * S + 5);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
  float *s_bias = (float *)(smem + S * CF::STAGE_BYTES + 256);
  uint8_t *s_slots = (uint8_t *)(s_bias + BN);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
  const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);
  const uint32_t mma_done = smem_u32(bars + 2 * S + 4);

  // rows and tiles (dense-path row count read from the device)
  int M = p.m_dev ? *p.m_dev : p.M_host;
  const bool dense_all = p.ctl ? p.ctl->dense != 0 : false;
  const int m_blocks = (M + BM - 1) / BM;
  const int n_blocks = (p.N + BN - 1) / BN;
  const int NQ = EPI == EPI_DW ? p.nq : 1;  // independent problems of one shape
  const int tiles_q = m_blocks * n_blocks;
  const int num_tiles = NQ * tiles_q;
  // The dense-path dx GEMM contracts over two K ranges of KT1 k-blocks:
  // dz with W_gate, then du with W_up (the plain FFN: the first only).
  const int Kd = p.k_dev ? *p.k_dev : p.Kdim;
  const int KT1 = (Kd + BK - 1) / BK;
  const int NR = (EPI == EPI_DX && p.gated) ? 2 : 1;
  const int KT = NR * KT1;
  // Tile order.  When B is larger than half of L2, groups of gm M-blocks,
  // and within a group all N-blocks with the M-blocks innermost: the CTAs in
  // flight then share a group's A rows (about 32 MB) and a few B tiles, and
  // each pass over B serves gm M-blocks from L2 (d_model 4096 / d_ff 14336:
  // B = W is 117 MB, streamed ~25 times per launch M-block by M-block,
  // twice grouped; gate GEMM 0.68 -> 0.53 ms).  A B that stays in L2 keeps
  // the plain M-block-major order (gm = 1), measured slightly faster there.
  const double b_bytes = (double)p.N * NB * BK * 2.0 * (double)KT;
  const int gm = b_bytes > 0.5 * (double)p.l2_bytes
                     ? max(1, min(m_blocks, (32 << 20) / (BM * 2 * BK * max(KT, 1))))
                     : 1;
  if ((int)blockIdx.x >= num_tiles || KT == 0) return;  // uniform for the CTA
  // EPI_DHS runs only when the dispatcher chose it (else the gather SDDMM)
  if (EPI == EPI_DHS && (dense_all || !p.ctl->dh_gemm)) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(CF::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      // all-dense mode reads the operand in place (a[1] / b[1]), otherwise
      // the gathered rows (a[0] / b[0])
      const CUtensorMap *amap0 = (EPI != EPI_DX && p.ctl && dense_all) ? &maps.a[1] : &maps.a[0];
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int q = tile / tiles_q;
        int mb, nb;
        tile_mn(tile - q * tiles_q, m_blocks, n_blocks, gm, mb, nb);
        // EPI_DW: this problem's A, and B = x (or dy for the last problem)
        const CUtensorMap *aq = EPI == EPI_DW ? &maps.a[q] : amap0;
        const int bq = (EPI == EPI_DW && q == NQ - 1) ? 2 : 0;
        for (int kt = 0; kt < KT; ++kt) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sbase = smem_u32(stages + stage * CF::STAGE_BYTES);
          const uint32_t fb = full0 + 8 * stage;
          mbar_expect_tx(fb, CF::STAGE_BYTES);
          const int r = NR > 1 ? kt / KT1 : 0;   // K range
          const int kc = (kt - r * KT1) * BK;     // k within the range
          const bool second = EPI == EPI_DX && r == 1;
          const CUtensorMap *amap = second ? &maps.a[1] : aq;
          if (A_MN) {
#pragma unroll
            for (int i = 0; i < BM / 64; ++i)
              tma_load_2d(sbase + i * (64 * BK * 2), amap, mb * BM + 64 * i, kc, fb);
          } else {
            tma_load_2d(sbase, amap, kc, mb * BM, fb);
          }
#pragma unroll
          for (int op = 0; op < NB; ++op) {
            const CUtensorMap *bm = &maps.b[bq + ((op == 1 || second) ? 1 : 0)];
            const uint32_t bbase = sbase + CF::A_BYTES + op * CF::B_BYTES;
            if (B_MN) {
#pragma unroll
              for (int i = 0; i < BN / 64; ++i)
                tma_load_2d(bbase + i * (64 * BK * 2), bm, nb * BN + 64 * i, kc, fb);
            } else {
              tma_load_2d(bbase, bm, kc, nb * BN, fb);
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain after an abort: wait (bounded) until the last load issued into
      // each stage has landed, so no copy is in flight when the CTA exits.
      if (!ok) {
        for (int s = 0; s < S && s < issued; ++s) {
          const long last = s + (long)S * ((issued - 1 - s) / S);
          const uint32_t par = (uint32_t)((last / S) & 1);
          const uint64_t t0 = global_timer();
          while (!mbar_try(full0 + 8 * s, par) && global_timer() - t0 < DRAIN_LIMIT_NS) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t IDESC = make_idesc(BM, BN, A_MN, B_MN, F16);
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++lt) {
        const int buf = lt & 1;
        const uint32_t use = (uint32_t)(lt >> 1);
        if (!mbar_wait(tempty0 + 8 * buf, (use & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t dacc = tmem_base + (uint32_t)(buf * NB * BN);
        for (int kt = 0; kt < KT; ++kt) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sbase = smem_u32(stages + stage * CF::STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // (an MN-major A tile is laid out as an MN-major B tile: see below)
            const uint64_t ad = A_MN ? sw128_desc(sbase + kk * 2048, 64 * BK * 2, 1024)
                                     : sw128_desc(sbase + kk * 32, 16, 1024);
#pragma unroll
            for (int op = 0; op < NB; ++op) {
              const uint32_t bbase = sbase + CF::A_BYTES + op * CF::B_BYTES;
              // K-major: 128 B rows, 8-row groups 1024 B apart, K step = +32 B.
              // MN-major: 64-element MN groups 8 KB apart (LBO), 8-row K groups
              // 1024 B apart (SBO), K step of 16 rows = +2048 B.
              const uint64_t bd = B_MN ? sw128_desc(bbase + kk * 2048, 64 * BK * 2, 1024)
                                       : sw128_desc(bbase + kk * 32, 16, 1024);
              mma_bf16(dacc + op * BN, ad, bd, IDESC, (kt > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * buf);
      }
      // All MMAs issued by this thread are complete before TMEM is freed.
      mma_commit(mma_done);
      const uint64_t t0 = global_timer();
      while (!mbar_try(mma_done, 0) && global_timer() - t0 < DRAIN_LIMIT_NS) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;          // accumulator row of this thread
    const int et = threadIdx.x - 64;        // 0..127 among epilogue threads
    // EPI_DHS with two 128-column TwELL tiles per output tile and K <= 8:
    // each row's slot data is fetched one output tile ahead (while the
    // previous tile is processed), so its latency is hidden even when the
    // epilogue, not the MMAs, sets the pace
    const bool pf2 = EPI == EPI_DHS && BN == 256 && p.C == 128 && p.Kslots <= 8;
    DhsSlots dcur, dnxt;
    auto dhs_fetch_tile = [&](int t_, DhsSlots &S) {
      int mb_, nb_;
      tile_mn(t_ - (t_ / tiles_q) * tiles_q, m_blocks, n_blocks, gm, mb_, nb_);
      const int m_ = mb_ * BM + row;
      dhs_fetch(p, m_, m_ < M, nb_ * BN, S);
    };
    if (pf2 && (int)blockIdx.x < num_tiles) dhs_fetch_tile(blockIdx.x, dcur);
    int lt = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++lt) {
      const int q = tile / tiles_q;
      int mb, nb;
      tile_mn(tile - q * tiles_q, m_blocks, n_blocks, gm, mb, nb);
      const int buf = lt & 1;
      const uint32_t use = (uint32_t)(lt >> 1);
      const int n0 = nb * BN;
      const int m = mb * BM + row;
      const bool row_ok = m < M;
      // per-tile column constants
      if (EPI == EPI_PACK || EPI == EPI_GU) {
        epi_bar();
        for (int c = et; c < BN; c += 128) s_bias[c] = (n0 + c < p.N) ? p.bg[n0 + c] : 0.f;
        epi_bar();
      }
      // EPI_U / EPI_DH: the slots of the tile's first TwELL tile are fetched
      // while the accumulator is still being computed (they do not depend on
      // it); EPI_DH also fetches u at the slots, and rows with a dense backup
      // row (ps >= 0) read that instead
      constexpr bool SLOTS = EPI == EPI_U || EPI == EPI_DH || EPI == EPI_DHS;
      const int tok_u = (SLOTS && row_ok) ? ((dense_all || EPI == EPI_DHS) ? m : p.rows[m]) : 0;
      const int ps_u = ((EPI == EPI_DH || (EPI == EPI_DHS && !pf2)) && row_ok) ? p.pos[tok_u] : -1;
      int pf_nz = 0;
      uint32_t pf_iw[8], pf_vw[16], pf_qw[16] = {};  // (pf_qw: plain FFN leaves it zero)
      if (pf2 && tile + (int)gridDim.x < num_tiles) dhs_fetch_tile(tile + gridDim.x, dnxt);
      if (SLOTS && row_ok && ps_u < 0 && !pf2) {
        fetch_slots(p, n0, tok_u, pf_nz, pf_iw, pf_vw);
        if ((EPI == EPI_DH || EPI == EPI_DHS) && p.gated)
          load_vals(p.uval + ((size_t)(n0 / p.C) * p.Tn + tok_u) * p.Kslots, p.Kslots, pf_qw);
      }
      // Each epilogue thread waits (bounded) for the accumulator; the AND of
      // the outcomes is taken at a barrier, so if any thread gave up (or
      // another role aborted) all four warps leave here together.
      const bool ok = epi_all(mbar_wait(tfull0 + 8 * buf, use & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * NB * BN);

      if (EPI == EPI_PACK) {
        const float rbv = (p.rb && row_ok) ? p.rb[m] : 0.f;
        const int K = p.Kslots;
        uint8_t *my_idx = s_slots + row * 32;
        bf16 *my_val = (bf16 *)(s_slots + 128 * 32) + row * 32;
        bf16 *my_z = (bf16 *)(s_slots + 128 * 32 * 3) + row * 32;
        uint32_t my_slots = 0;  // slots this row writes in this output tile
        for (int jt = 0; jt < BN / p.C; ++jt) {
          const int j = (n0 + jt * p.C) / p.C;      // global TwELL tile index
          const bool tile_ok = n0 + jt * p.C < p.N;
          for (int k = 0; k < K; ++k) {
            my_idx[k] = 0xFF;
            my_val[k] = __float2bfloat16_rn(0.f);
          }
          // Per 32-column block: z and its activity mask without branches (a
          // branch per value serialised the add -> compare -> branch chain of
          // the one epilogue warp per SM sub-partition); only a block with an
          // active column (about a quarter of them at 1% density) stages its
          // bf16 values and appends the active columns in ascending order.
          int cnt = 0;
          for (int c0 = 0; c0 < p.C; c0 += 32) {
            float v[32];
            tmem_ld32(tacc + jt * p.C + c0, v);
            const float *bb = s_bias + jt * p.C + c0;
            uint32_t msk = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v[i] = (v[i] + bb[i]) + rbv;  // z
              msk |= (v[i] > 0.f ? 1u : 0u) << i;
            }
            if (msk) {
#pragma unroll
              for (int i = 0; i < 32; i += 8)
                *(uint4 *)(my_z + i) = make_uint4(pack_bf2(v[i], v[i + 1]), pack_bf2(v[i + 2], v[i + 3]),
                                                  pack_bf2(v[i + 4], v[i + 5]), pack_bf2(v[i + 6], v[i + 7]));
              do {
                const int b = __ffs(msk) - 1;
                msk &= msk - 1;
                if (cnt < K) {
                  my_idx[cnt] = (uint8_t)(c0 + b);
                  my_val[cnt] = my_z[b];
                }
                ++cnt;
              } while (msk);
            }
          }
          if (row_ok && tile_ok) {
            const size_t s0 = ((size_t)j * p.Tn + m) * (size_t)K;
            uint8_t *gi = p.idx + s0;
            bf16 *gv = p.val + s0;
            if (K % 16 == 0) {
              for (int k = 0; k < K; k += 16) *(uint4 *)(gi + k) = *(const uint4 *)(my_idx + k);
            } else if (K == 8) {
              *(uint2 *)gi = *(const uint2 *)my_idx;
            } else if (K == 4) {
              *(uint32_t *)gi = *(const uint32_t *)my_idx;
            } else {
              for (int k = 0; k < K; ++k) gi[k] = my_idx[k];
            }
            if (K % 8 == 0) {
              for (int k = 0; k < K; k += 8) *(uint4 *)(gv + k) = *(const uint4 *)(my_val + k);
            } else {
              for (int k = 0; k < K; ++k) gv[k] = my_val[k];
            }
            p.nnz[(size_t)j * p.Tn + m] = (uint8_t)cnt;
            if (cnt > K) atomicOr(&p.ovf_bits[m >> 5], 1u << (m & 31));
            my_slots += (uint32_t)(cnt < K ? cnt : K);
          }
          // An overflowing (row, tile) also keeps its full ReLU(z) tile (the
          // accumulator is read again; the load is warp-collective).
          const bool wide_row = row_ok && tile_ok && cnt > K;
          if (__any_sync(0xffffffffu, wide_row)) {
            for (int c0 = 0; c0 < p.C; c0 += 32) {
              float v[32];
              tmem_ld32(tacc + jt * p.C + c0, v);
              if (!wide_row) continue;
              uint32_t wv[16];
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float z0 = (v[i] + s_bias[jt * p.C + c0 + i]) + rbv;
                const float z1 = (v[i + 1] + s_bias[jt * p.C + c0 + i + 1]) + rbv;
                wv[i / 2] = pack_bf2(z0 > 0.f ? z0 : 0.f, z1 > 0.f ? z1 : 0.f);
              }
              uint4 *wd = (uint4 *)(p.wide + ((size_t)j * p.Tn + m) * p.C + c0);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                wd[v4] = make_uint4(wv[4 * v4], wv[4 * v4 + 1], wv[4 * v4 + 2], wv[4 * v4 + 3]);
            }
          }
        }
        const uint32_t warp_slots = __reduce_add_sync(0xffffffffu, my_slots);
        if (lane == 0 && warp_slots && p.slots) atomicAdd(p.slots, (unsigned long long)warp_slots);
      } else if (EPI == EPI_GU) {
        const int tok = row_ok ? (dense_all ? m : p.rows[m]) : 0;
        const float rbv = (p.rb && row_ok) ? p.rb[tok] : 0.f;
        const int ps = row_ok ? (dense_all ? p.pos[tok] : m) : -1;
        const bool fb_ok = ps >= 0 && ps < p.cap;
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float zg[32], zu[32];
          tmem_ld32(tacc + c0, zg);
          if (NB == 2) tmem_ld32(tacc + BN + c0, zu);
          if (!row_ok || n0 + c0 >= p.N) continue;
          uint32_t hw[16], gw[16], uw[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float g2[2], u2[2], h2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float z = (zg[i + e] + s_bias[c0 + i + e]) + rbv;
              g2[e] = z > 0.f ? __bfloat162float(__float2bfloat16_rn(z)) : 0.f;
              u2[e] = NB == 2 ? zu[i + e] : 1.f;
              h2[e] = p.gated ? g2[e] * u2[e] : g2[e];
            }
            hw[i / 2] = pack_bf2(h2[0], h2[1]);
            gw[i / 2] = pack_bf2(g2[0], g2[1]);
            uw[i / 2] = pack_bf2(u2[0], u2[1]);
          }
          uint4 *hd = (uint4 *)(p.h + (size_t)m * p.F + n0 + c0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            hd[v4] = make_uint4(hw[4 * v4], hw[4 * v4 + 1], hw[4 * v4 + 2], hw[4 * v4 + 3]);
          if (fb_ok) {
            uint4 *gd = (uint4 *)(p.g_fb + (size_t)ps * p.F + n0 + c0);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              gd[v4] = make_uint4(gw[4 * v4], gw[4 * v4 + 1], gw[4 * v4 + 2], gw[4 * v4 + 3]);
            if (p.train && p.gated) {
              uint4 *ud = (uint4 *)(p.u_fb + (size_t)ps * p.F + n0 + c0);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                ud[v4] = make_uint4(uw[4 * v4], uw[4 * v4 + 1], uw[4 * v4 + 2], uw[4 * v4 + 3]);
            }
          }
        }
      } else if (EPI == EPI_U) {
        // Dense-path rows of the gated FFN with B = W_up only: g is not
        // recomputed but read back from what the gate epilogue stored (the
        // bf16 value of every active entry: the wide tile of an overflowing
        // (row, tile), else the TwELL slots), so this GEMM does half the work
        // of the gate + up one.  The slots of the next TwELL tile are fetched
        // while the current one is processed; each 32-column block scatters
        // them branch-free (an entry outside the block goes to a spare
        // element).  Stores h and the backup rows as EPI_GU; in all-dense
        // training also u at the slots of the non-overflow rows.
        const int tok = tok_u;
        const int ps = row_ok ? (dense_all ? p.pos[tok] : m) : -1;
        const bool fb_ok = ps >= 0 && ps < p.cap;
        const int K = p.Kslots;
        bf16 *gz = (bf16 *)s_slots + row * GZ_STRIDE;  // this row's g for the current 32 columns
        const int n_end = min(n0 + BN, p.N);
        int nz = 0;
        uint32_t iw[8], vw[16];
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float zu[32];
          tmem_ld32(tacc + c0, zu);
          if (!row_ok || n0 + c0 >= p.N) continue;
          const int cl = (n0 + c0) % p.C;
          if (cl == 0) {  // a new TwELL tile: take the fetched slots, fetch the next tile's
            nz = pf_nz;
#pragma unroll
            for (int i = 0; i < 8; ++i) iw[i] = pf_iw[i];
#pragma unroll
            for (int i = 0; i < 16; ++i) vw[i] = pf_vw[i];
            if (n0 + c0 + p.C < n_end) fetch_slots(p, n0 + c0 + p.C, tok, pf_nz, pf_iw, pf_vw);
          }
          if (nz > K) {
            const size_t jt = (size_t)((n0 + c0) / p.C) * p.Tn + tok;
            const uint4 *wr = (const uint4 *)(p.wide + jt * p.C + cl);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) ((uint4 *)gz)[v4] = wr[v4];
          } else {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) ((uint4 *)gz)[v4] = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              if (k >= K) break;  // uniform
              const int c = slot_col(iw, k) - cl;
              const bool in = k < nz && (unsigned)c < 32u;
              gz[in ? c : 32] = __ushort_as_bfloat16(slot_val(vw, k));
            }
          }
          uint32_t uw[16];
          float hv[32];
          const uint4 *g4 = (const uint4 *)gz;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const uint4 gv = g4[v4];
            const uint32_t gp[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
              const int i = 8 * v4 + 2 * q2;
              hv[i] = bf_lo(gp[q2]) * zu[i];
              hv[i + 1] = bf_hi(gp[q2]) * zu[i + 1];
              uw[i / 2] = pack_bf2(zu[i], zu[i + 1]);
            }
          }
          // h = g u (fp32) as the fp16 operand of the down GEMM
          store_f16x32((__half *)p.h + (size_t)m * p.F + n0 + c0, hv, p.status);
          if (dense_all && p.train && ps < 0) {
            // all-dense training: u at this row's slots in the block (staged
            // in shared memory to be picked by slot column)
            bf16 *uz = (bf16 *)s_slots + 128 * GZ_STRIDE + row * 32;
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              ((uint4 *)uz)[v4] = make_uint4(uw[4 * v4], uw[4 * v4 + 1], uw[4 * v4 + 2], uw[4 * v4 + 3]);
            const size_t s0 = ((size_t)((n0 + c0) / p.C) * p.Tn + tok) * K;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              if (k >= K) break;  // uniform
              const int c = slot_col(iw, k) - cl;
              if (k < nz && (unsigned)c < 32u) p.uval[s0 + k] = uz[c];
            }
          }
          if (fb_ok) {
            uint4 *gd = (uint4 *)(p.g_fb + (size_t)ps * p.F + n0 + c0);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) gd[v4] = g4[v4];
            if (p.train) {
              uint4 *ud = (uint4 *)(p.u_fb + (size_t)ps * p.F + n0 + c0);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                ud[v4] = make_uint4(uw[4 * v4], uw[4 * v4 + 1], uw[4 * v4 + 2], uw[4 * v4 + 3]);
            }
          }
        }
      } else if (EPI == EPI_DH) {
        // Backward of the dense-path rows.  g and u of the row come from what
        // the forward saved: the dense backup rows of an overflow row, else
        // the TwELL slots (g) and u at the slots, loaded once per tile with
        // vector loads.  dz, du and h = g u are computed in fp32 and stored
        // as fp16 rows (the operands of the dx and weight-gradient GEMMs) at
        // row m of p.dz2 / p.du2 / p.h2.  Rows past the last one (inside this
        // tile) are written as zeros: the weight-gradient GEMMs contract over
        // them.
        const int tok = tok_u;
        const int ps = ps_u;
        const int K = p.Kslots;
        bf16 *gz = (bf16 *)s_slots + row * 2 * GZ_STRIDE, *uz = gz + GZ_STRIDE;  // g, u of 32 columns
        // (one set of slot registers: the first TwELL tile's were fetched
        // before the accumulator wait, a later tile's are fetched when the
        // tile starts; two sets would not fit the register budget)
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(tacc + c0, v);
          if (n0 + c0 >= p.N) continue;  // uniform (F is a multiple of 32)
          const size_t o = (size_t)m * p.F + n0 + c0;
          float dz[32], du[32], hv[32];
          if (row_ok) {
            uint32_t ga[16], ua[16];  // bf16 pairs of g and u (plain FFN: u = 1)
            if (ps >= 0) {  // overflow row: backup rows (none past the capacity: zeros)
              const bool ok = ps < p.cap;
              const uint4 *gr = (const uint4 *)(p.g_fb + (size_t)ps * p.F + n0 + c0);
              const uint4 *ur = (const uint4 *)(p.u_fb + (size_t)ps * p.F + n0 + c0);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                const uint4 gv = ok ? gr[v4] : make_uint4(0, 0, 0, 0);
                const uint4 uv = (ok && p.gated) ? ur[v4] : make_uint4(0, 0, 0, 0);
                ga[4 * v4] = gv.x; ga[4 * v4 + 1] = gv.y; ga[4 * v4 + 2] = gv.z; ga[4 * v4 + 3] = gv.w;
                ua[4 * v4] = uv.x; ua[4 * v4 + 1] = uv.y; ua[4 * v4 + 2] = uv.z; ua[4 * v4 + 3] = uv.w;
              }
            } else {  // slots (every tile of the row holds at most K)
              const int cl = (n0 + c0) % p.C;
              if (cl == 0 && c0 > 0) {  // a later TwELL tile
                fetch_slots(p, n0 + c0, tok, pf_nz, pf_iw, pf_vw);
                if (p.gated)
                  load_vals(p.uval + ((size_t)((n0 + c0) / p.C) * p.Tn + tok) * K, K, pf_qw);
              }
              const int nz = min(pf_nz, K);
              if (cl == 0) {  // a malformed live slot (index >= C) lands in no block
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                  if (k >= K) break;  // uniform
                  if (k < nz && slot_col(pf_iw, k) >= p.C) set_status(p.status, TWELL_ERR_INDEX);
                }
              }
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                ((uint4 *)gz)[v4] = make_uint4(0, 0, 0, 0);
                ((uint4 *)uz)[v4] = make_uint4(0, 0, 0, 0);
              }
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                if (k >= K) break;  // uniform
                const int c = slot_col(pf_iw, k) - cl;
                const int e = (k < nz && (unsigned)c < 32u) ? c : 32;  // 32: spare element
                gz[e] = __ushort_as_bfloat16(slot_val(pf_vw, k));
                uz[e] = __ushort_as_bfloat16(slot_val(pf_qw, k));
              }
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                const uint4 gv = ((const uint4 *)gz)[v4], uv = ((const uint4 *)uz)[v4];
                ga[4 * v4] = gv.x; ga[4 * v4 + 1] = gv.y; ga[4 * v4 + 2] = gv.z; ga[4 * v4 + 3] = gv.w;
                ua[4 * v4] = uv.x; ua[4 * v4 + 1] = uv.y; ua[4 * v4 + 2] = uv.z; ua[4 * v4 + 3] = uv.w;
              }
            }
            if (!p.gated) {
#pragma unroll
              for (int i = 0; i < 16; ++i) ua[i] = 0x3F803F80u;  // u = 1
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float g = (i & 1) ? bf_hi(ga[i / 2]) : bf_lo(ga[i / 2]);
              const float u = (i & 1) ? bf_hi(ua[i / 2]) : bf_lo(ua[i / 2]);
              const float h = p.gated ? g * u : g;
              const float dh = v[i] + p.lambda * (h > 0.f ? 1.f : (h < 0.f ? -1.f : 0.f));
              const bool act = g > 0.f;
              dz[i] = act ? (p.gated ? dh * u : dh) : 0.f;
              du[i] = act ? dh * g : 0.f;
              hv[i] = h;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) dz[i] = du[i] = hv[i] = 0.f;
          }
          store_f16x32(p.dz2 + o, dz, p.status);
          if (p.gated) store_f16x32(p.du2 + o, du, p.status);
          store_f16x32(p.h2 + o, hv, p.status);
          // dbg: column sums of this warp's 32 rows by recursive halving (lane
          // l ends with column l), stored per 32-row group (m / 32) and
          // summed in group order by the weight-gradient GEMM: no atomics,
          // so the sum is the same on every run
#pragma unroll
          for (int w = 16; w >= 1; w >>= 1) {
            const bool up = (lane & w) != 0;
#pragma unroll
            for (int i = 0; i < w; ++i) {
              const float send = up ? dz[i] : dz[i + w];
              const float keep = up ? dz[i + w] : dz[i];
              dz[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
            }
          }
          p.dbg_r[(size_t)(m >> 5) * p.F + n0 + c0 + lane] = dz[0];
        }
      } else if (EPI == EPI_DHS) {
        // dh of the rows the gathers own (not the dense-path rows), from the
        // full product dy W_down^T but read only where the forward kept an
        // active entry: at the row's TwELL slots (through the thread's
        // shared-memory row, 32 columns at a time, only for blocks that hold
        // a slot), or at every column of an overflow row with a dense backup
        // row; then the gradients of each entry as the gather SDDMM stores
        // them.  With two 128-column TwELL tiles and K <= 8 the slots of
        // both are prefetched before the accumulator wait, every accumulator
        // column is read, and the TMEM buffer is released before the slot
        // gradients are computed and stored.  (Measured on the d_model 2048 /
        // d_ff 8192 step: with a drain-only epilogue the kernel takes 78 us,
        // and the epilogue's global loads and its stores each add about
        // 11 us although the epilogue overlaps the next tile's MMAs, so only
        // live slots are stored: 102.6 -> 99.0 us.)
        const int tok = m;
        const int ps = pf2 ? dcur.ps : ps_u;
        const bool skip = !row_ok || ps >= p.cap || (ps >= 0 && p.ctl->ovf_gemm);
        const int K = p.Kslots;
        float *st = (float *)s_slots + row * DHS_STRIDE;
        const int nch = (p.Tn + TR_CHUNK - 1) / TR_CHUNK;
        if (pf2) {
          const bool two = n0 + 128 < p.N;  // uniform: the second TwELL tile exists
          const int nz0 = min(dcur.nz0, K), nz1 = min(dcur.nz1, K);
          const uint32_t blk =
              dhs_blocks<8>(dcur.i0, K, nz0, 128) | (dhs_blocks<8>(dcur.i1, K, nz1, 128) << 4);
          float d0[8], d1[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) d0[k] = d1[k] = 0.f;
#pragma unroll 1
          for (int cb = 0; cb < 256; cb += 32) {
            if (cb >= 128 && !two) break;  // uniform
            float v[32];
            tmem_ld32(tacc + cb, v);  // (warp-collective)
            if (skip) continue;
            if (ps >= 0) dhs_store_row_block(p, ps, n0 + cb, v);
            else if ((blk >> (cb >> 5)) & 1u) {
              if (cb < 128) dhs_pick<8>(st, v, cb, K, nz0, dcur.i0, d0);
              else dhs_pick<8>(st, v, cb - 128, K, nz1, dcur.i1, d1);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty0 + 8 * buf);
          if (!skip && ps < 0) {
            dhs_store_slots<8>(p, n0 / 128, tok, K, nz0, dcur.i0, dcur.v0, dcur.q0, d0, nch);
            if (two)
              dhs_store_slots<8>(p, n0 / 128 + 1, tok, K, nz1, dcur.i1, dcur.v1, dcur.q1, d1, nch);
          }
          dcur = dnxt;  // the next tile's slots (fetched before this tile's wait)
          continue;     // the buffer is released
        }
        for (int jt = 0; jt < BN / p.C; ++jt) {
          const int n1 = n0 + jt * p.C;
          if (n1 >= p.N) break;  // uniform
          if (jt > 0 && !skip && ps < 0) {  // the first tile's slots were prefetched
            fetch_slots(p, n1, tok, pf_nz, pf_iw, pf_vw);
            if (p.gated) load_vals(p.uval + ((size_t)(n1 / p.C) * p.Tn + tok) * K, K, pf_qw);
          }
          const int nz = min(pf_nz, K);
          const uint32_t blk = dhs_blocks<32>(pf_iw, K, nz, p.C);
          float dhv[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) dhv[k] = 0.f;
          for (int cb = 0; cb < p.C; cb += 32) {
            float v[32];
            tmem_ld32(tacc + jt * p.C + cb, v);  // (warp-collective)
            if (skip) continue;
            if (ps >= 0) dhs_store_row_block(p, ps, n1 + cb, v);
            else if ((blk >> (cb >> 5)) & 1u) dhs_pick<32>(st, v, cb, K, nz, pf_iw, dhv);
          }
          if (skip || ps >= 0) continue;
          dhs_store_slots<32>(p, n1 / p.C, tok, K, nz, pf_iw, pf_vw, pf_qw, dhv, nch);
        }
      } else if (EPI == EPI_DW) {
        // Weight-gradient rows (row m = neuron, fp32) of problem q: stored
        // in all-dense mode, added to the gather kernel's rows otherwise.
        float *out = p.outq[q];
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(tacc + c0, v);
          if (!row_ok || n0 + c0 >= p.N) continue;
          float *o = out + (size_t)m * p.N + n0 + c0;
          if (n0 + c0 + 32 > p.N) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (n0 + c0 + i < p.N) o[i] = dense_all ? v[i] : o[i] + v[i];
            continue;
          }
          float4 *o4 = (float4 *)o;
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            float4 r = make_float4(v[4 * v4], v[4 * v4 + 1], v[4 * v4 + 2], v[4 * v4 + 3]);
            if (!dense_all) {
              const float4 q4 = o4[v4];
              r.x += q4.x; r.y += q4.y; r.z += q4.z; r.w += q4.w;
            }
            o4[v4] = r;
          }
        }
        if (q == 0 && nb == 0 && row_ok) {  // dbg: the dense-path rows' group sums, in order
          const int groups = (*p.k_dev + 127) / 128 * 4;
          float sb = 0.f;
          for (int g = 0; g < groups; ++g) sb += p.dbg_r[(size_t)g * p.F + m];
          p.dbg_out[m] = (dense_all ? 0.f : p.dbg_out[m]) + sb;
        }
      } else if (EPI == EPI_DOWN || EPI == EPI_DX) {
        const int tok = row_ok ? (dense_all ? m : p.rows[m]) : 0;
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(tacc + c0, v);
          if (!row_ok || n0 + c0 >= p.N) continue;
          if (n0 + c0 + 32 > p.N) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (n0 + c0 + i < p.N) p.y[(size_t)tok * p.D + n0 + c0 + i] = __float2bfloat16_rn(v[i]);
            continue;
          }
          uint4 *yd = (uint4 *)(p.y + (size_t)tok * p.D + n0 + c0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            yd[v4] = make_uint4(pack_bf2(v[8 * v4], v[8 * v4 + 1]), pack_bf2(v[8 * v4 + 2], v[8 * v4 + 3]),
                                pack_bf2(v[8 * v4 + 4], v[8 * v4 + 5]),
                                pack_bf2(v[8 * v4 + 6], v[8 * v4 + 7]));
        }
      } else {  // EPI_F32
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(tacc + c0, v);
          if (!row_ok) continue;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (n0 + c0 + i < p.N) p.out[(size_t)m * p.N + n0 + c0 + i] = v[i];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * buf);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(CF::TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host --
long long l2_size() {
  static long long n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) == cudaSuccess && v > 0) n = v;
  });
  return n;
}

int gather_passes(int requested, double set_bytes, int nv, int min_width) {
  int n = requested;
  if (n <= 0) {  // automatic: passes whose working sets fit in GATHER_L2_SHARE of L2
    const double budget = GATHER_L2_SHARE * (double)l2_size();
    n = 1;
    while (budget > 0.0 && set_bytes / n > budget && n < GATHER_MAX_PASSES &&
           nv / (2 * n) >= min_width)
      n *= 2;
  }
  if (n > nv) n = nv;
  return n < 1 ? 1 : n;
}

int num_sms() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  });
  return n;
}

namespace {

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeFn)f;
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix, box {bc, br},
// 128-byte swizzle (bc * 2 == 128).
bool make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t bc,
              uint32_t br) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {bc, br};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int BN, int NB, bool B_MN, int EPI, bool A_MN = false, bool F16 = false>
cudaError_t launch_tc(const TcMaps &maps, const TcParams &p, int max_tiles, cudaStream_t s) {
  using CF = Cfg<BN, NB, B_MN, EPI, A_MN>;
  auto kern = tc_gemm_kernel<BN, NB, B_MN, EPI, A_MN, F16>;
  // once per instantiation and process (concurrent first calls from several
  // host threads are safe)
  static cudaError_t attr_err = cudaSuccess;
  static std::once_flag attr_once;
  std::call_once(attr_once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  int grid = max_tiles < num_sms() ? max_tiles : num_sms();
  if (grid < 1) grid = 1;
  TcParams q = p;
  q.l2_bytes = l2_size();
  launch_k(kern, grid, NTHREADS, CF::SMEM, s, maps, q);
  return cudaGetLastError();
}

template <int BN, int NB, bool B_MN, int EPI, bool A_MN = false, bool F16 = false>
cudaError_t launch_tc(const CUtensorMap &a, const CUtensorMap &a2, const CUtensorMap &b0,
                      const CUtensorMap &b1, const TcParams &p, int max_tiles, cudaStream_t s) {
  TcMaps maps;
  maps.a[0] = a; maps.a[1] = a2; maps.a[2] = a;
  maps.b[0] = b0; maps.b[1] = b1; maps.b[2] = b0; maps.b[3] = b1;
  return launch_tc<BN, NB, B_MN, EPI, A_MN, F16>(maps, p, max_tiles, s);
}

TcParams base_params(const FwdArgs &a) {
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.Tn = a.T; p.F = a.F; p.D = a.D; p.C = a.C; p.Kslots = a.K; p.cap = a.tw.ovf_cap;
  p.gated = a.gated; p.train = a.train; p.bg = a.bg; p.rb = a.rb; p.rows = a.ws.rows;
  p.pos = a.ws.pos; p.idx = a.tw.idx; p.nnz = a.tw.nnz; p.val = (bf16 *)a.tw.val;
  p.uval = (bf16 *)a.tw.u_val;
  p.ovf_bits = a.ws.ovf_bits;
  p.slots = &a.ws.ctl->slots;
  p.wide = (bf16 *)a.ws.wide;
  p.h = (bf16 *)a.ws.h; p.g_fb = (bf16 *)a.tw.g_fb; p.u_fb = (bf16 *)a.tw.u_fb; p.y = (bf16 *)a.y;
  p.status = a.tw.status;
  p.Tp = a.ws.rp;  // rows of the h hi part (the lo part follows)
  return p;
}

}  // namespace

bool tc_available() {
  static int ok = -1;
  if (ok < 0) {
    int dev = 0, major = 0, minor = 0;
    ok = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess)
      ok = (major == 10 && minor == 3 && encode_fn() != nullptr) ? 1 : 0;
  }
  return ok == 1;
}

cudaError_t launch_tc_gate_pack(const FwdArgs &a, cudaStream_t s) {
  CUtensorMap mx, mw;
  // 128 x 256 output tiles: each A tile feeds twice the MMA work of a
  // 128 x 128 tile, which halves the A re-reads and the shared-memory
  // operand traffic per flop.
  constexpr int GBN = 256;
  if (!make_map(&mx, a.x, a.D, a.T, 64, BM) || !make_map(&mw, a.Wg, a.D, a.F, 64, GBN))
    return cudaErrorInvalidValue;
  TcParams p = base_params(a);
  p.M_host = a.T;
  p.N = a.F;
  p.Kdim = a.D;
  const int tiles = ((a.T + BM - 1) / BM) * ((a.F + GBN - 1) / GBN);
  return launch_tc<GBN, 1, false, EPI_PACK>(mx, mx, mw, mw, p, tiles, s);
}

cudaError_t launch_tc_dense_gu(const FwdArgs &a, cudaStream_t s) {
  CUtensorMap mxg, mx, mg, mu;
  if (!make_map(&mxg, a.ws.xg, a.D, a.T, 64, BM) || !make_map(&mx, a.x, a.D, a.T, 64, BM) ||
      !make_map(&mg, a.Wg, a.D, a.F, 64, 128) ||
      !make_map(&mu, a.gated ? a.Wu : a.Wg, a.D, a.F, 64, 128))
    return cudaErrorInvalidValue;
  TcParams p = base_params(a);
  p.m_dev = &a.ws.ctl->n_rows;
  p.ctl = a.ws.ctl;
  p.N = a.F;
  p.Kdim = a.D;
  if (a.gated) {  // up only (g from the stored TwELL / wide tiles), 128 x 256 tiles
    CUtensorMap mu256;
    if (!make_map(&mu256, a.Wu, a.D, a.F, 64, 256)) return cudaErrorInvalidValue;
    const int tiles = ((a.T + BM - 1) / BM) * ((a.F + 255) / 256);
    return launch_tc<256, 1, false, EPI_U>(mxg, mx, mu256, mu256, p, tiles, s);
  }
  const int tiles = ((a.T + BM - 1) / BM) * ((a.F + 127) / 128);
  return launch_tc<128, 1, false, EPI_GU>(mxg, mx, mg, mg, p, tiles, s);
}

// Down projection of the dense-path rows: A = h rows (dense-path order),
// B = W_down read MN-major from its neuron-major [F][D] storage.  Gated FFN:
// h (fp32 g u) and W_down in fp16 (its copy in the workspace); plain FFN:
// h = g, exact in bf16, against W_down itself.
cudaError_t launch_tc_dense_down(const FwdArgs &a, cudaStream_t s) {
  // 128 x 256 output tiles (as the gate GEMM): half the A re-reads of 128 x 128
  const int Tp = a.ws.rp;  // rows of the dense-path row buffers
  CUtensorMap mh, md;
  if (!make_map(&mh, a.ws.h, a.F, Tp, 64, BM) ||
      !make_map(&md, a.gated ? a.ws.wd16 : a.Wd, a.D, a.F, 64, 64))
    return cudaErrorInvalidValue;
  TcParams p = base_params(a);
  p.m_dev = &a.ws.ctl->n_rows;
  p.ctl = a.ws.ctl;
  p.N = a.D;
  p.Kdim = a.F;
  const int tiles = ((a.T + BM - 1) / BM) * ((a.D + 255) / 256);
  if (a.gated) return launch_tc<256, 1, true, EPI_DOWN, false, true>(mh, mh, md, md, p, tiles, s);
  return launch_tc<256, 1, true, EPI_DOWN>(mh, mh, md, md, p, tiles, s);
}

// ---------------------------------------------------------------------------
// Backward of the dense-path rows: every row in all-dense mode, else the
// overflow rows when there are at least OVF_GEMM_MIN of them (the kernels
// return at once when there are none).  Row buffers (Tp = ws.rp rows: T, or
// the caller's dense-row cap, rounded up to 128): ws.dzr / ws.dur / ws.hr =
// dz / du / h as bf16 hi rows then lo rows ([2 Tp][F]); ws.dyg / ws.xg =
// gathered dy / x rows ([Tp][D]).
namespace {

TcParams bwd_params(const BwdArgs &a) {
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.Tn = a.T; p.F = a.F; p.D = a.D; p.C = a.C; p.Kslots = a.K; p.cap = a.tw.ovf_cap;
  p.gated = a.gated; p.train = 1; p.rows = a.ws.rows; p.pos = a.ws.pos; p.ctl = a.ws.ctl;
  p.idx = a.tw.idx; p.nnz = a.tw.nnz; p.val = (bf16 *)a.tw.val; p.uval = (bf16 *)a.tw.u_val;
  p.g_fb = (bf16 *)a.tw.g_fb; p.u_fb = (bf16 *)a.tw.u_fb;
  p.dz2 = (__half *)a.ws.dzr; p.du2 = (__half *)a.ws.dur; p.h2 = (__half *)a.ws.hr;
  p.Tp = a.ws.rp;
  p.y = (bf16 *)a.dx; p.lambda = a.lambda; p.dbg_r = a.ws.dbg_r; p.status = a.tw.status;
  return p;
}

}  // namespace

// dh = dy W_down^T over the dense-path rows, then the L1 term and dz / du / h.
// fp16 operands: the dense-path dy rows (copied by the row-preparation
// kernel in every mode) and the workspace's fp16 copy of W_down, both exact
// copies of the bf16 values, so dh is the bf16 product's.
cudaError_t launch_tc_bwd_dh(const BwdArgs &a, cudaStream_t s) {
  const int Tp = a.ws.rp;  // rows of the dense-path row buffers
  CUtensorMap mdyg, mwd;
  if (!make_map(&mdyg, a.ws.dyg, a.D, Tp, 64, BM) || !make_map(&mwd, a.ws.wd16, a.D, a.F, 64, 256))
    return cudaErrorInvalidValue;
  TcParams p = bwd_params(a);
  p.m_dev = &a.ws.ctl->n_rows;
  p.N = a.F;
  p.Kdim = a.D;
  return launch_tc<256, 1, false, EPI_DH, false, true>(mdyg, mdyg, mwd, mwd, p,
                                                       (Tp / BM) * ((a.F + 255) / 256), s);
}

// dh of the rows the gathers own as one GEMM over every row, dy W_down^T
// (both K-major, 128 x 256 tiles as the gate GEMM), read at the TwELL slots
// by the epilogue: at ~1% active entries the tensor cores compute the whole
// product sooner than the SDDMM gathers a d_model row of W_down per entry.
cudaError_t launch_tc_bwd_dh_sampled(const BwdArgs &a, cudaStream_t s) {
  CUtensorMap mdy, mwd;
  if (!make_map(&mdy, a.dy, a.D, a.T, 64, BM) || !make_map(&mwd, a.Wd, a.D, a.F, 64, 256))
    return cudaErrorInvalidValue;
  TcParams p = bwd_params(a);
  p.M_host = a.T;
  p.N = a.F;
  p.Kdim = a.D;
  p.sdz = a.ws.dz; p.sdu = a.ws.du; p.shs = a.ws.hs;
  p.rdz = a.ws.dzr; p.rdu = a.ws.dur; p.rhs = a.ws.hr;
  p.col_chunk = a.ws.col_chunk;
  const int tiles = ((a.T + BM - 1) / BM) * ((a.F + 255) / 256);
  return launch_tc<256, 1, false, EPI_DHS>(mdy, mdy, mwd, mwd, p, tiles, s);
}

// dx[tok] = dz W_gate + du W_up over the dense-path rows (one accumulator,
// two K ranges; fp16 dz, du and the workspace's fp16 copies of W_gate,
// W_up, read MN-major from [F][D]).
cudaError_t launch_tc_bwd_dx(const BwdArgs &a, cudaStream_t s) {
  const int Tp = a.ws.rp;  // rows of the dense-path row buffers
  CUtensorMap mz, mu, mwg, mwu;
  if (!make_map(&mz, a.ws.dzr, a.F, Tp, 64, BM) || !make_map(&mu, a.ws.dur, a.F, Tp, 64, BM) ||
      !make_map(&mwg, a.ws.wg16, a.D, a.F, 64, 64) ||
      !make_map(&mwu, a.gated ? a.ws.wu16 : a.ws.wg16, a.D, a.F, 64, 64))
    return cudaErrorInvalidValue;
  TcParams p = bwd_params(a);
  p.m_dev = &a.ws.ctl->n_rows;
  p.N = a.D;
  p.Kdim = a.F;
  return launch_tc<256, 1, true, EPI_DX, false, true>(mz, mu, mwg, mwu, p,
                                                      (Tp / BM) * ((a.D + 255) / 256), s);
}

// dWg = dz^T x (+ dbg), dWu = du^T x, dWd = h^T dy over the dense-path rows:
// both operands MN-major, the token axis is the contraction; fp16 dz, du, h
// and the dense-path x, dy rows in fp16 (copied by the row-preparation kernel
// in every mode).  Stored in all-dense mode, added to the gather kernel's
// rows otherwise.
cudaError_t launch_tc_bwd_dw(const BwdArgs &a, cudaStream_t s) {
  const int Tp = a.ws.rp;  // rows of the dense-path row buffers
  // problems: dWg (A = dz, B = x), [dWu (du, x),] dWd (h, dy)
  TcMaps maps;
  const void *A[3] = {a.ws.dzr, a.gated ? (const void *)a.ws.dur : a.ws.hr, a.ws.hr};
  for (int q = 0; q < 3; ++q)
    if (!make_map(&maps.a[q], A[q], a.F, Tp, 64, 64)) return cudaErrorInvalidValue;
  if (!make_map(&maps.b[0], a.ws.xg, a.D, Tp, 64, 64) ||
      !make_map(&maps.b[2], a.ws.dyg, a.D, Tp, 64, 64))
    return cudaErrorInvalidValue;
  maps.b[1] = maps.b[0];
  maps.b[3] = maps.b[2];
  TcParams p = bwd_params(a);
  p.k_dev = &a.ws.ctl->n_rows;
  p.M_host = a.F;
  p.N = a.D;
  p.nq = a.gated ? 3 : 2;
  p.outq[0] = a.dWg;
  p.outq[1] = a.gated ? a.dWu : a.dWd;
  p.outq[2] = a.dWd;
  p.dbg_out = a.dbg;
  const int tiles = p.nq * ((a.F + BM - 1) / BM) * ((a.D + 255) / 256);
  return launch_tc<256, 1, true, EPI_DW, true, true>(maps, p, tiles, s);
}

#ifdef TWELL_TEST_HOOKS
// Test hook (built only into the test-hooks library, never into
// libtwell.so): fp32 C[M][N] = op(A) op(B), bf16 operands.  layout bit 0: B
// is [K][N] (MN-major), else [N][K]; bit 1: A is [K][M] (MN-major), else
// [M][K].
cudaError_t tc_test_gemm(const void *A, const void *B, float *Cout, int M, int N, int K, int layout,
                         int32_t *status, cudaStream_t s) {
  const bool b_mn = (layout & 1) != 0, a_mn = (layout & 2) != 0;
  CUtensorMap ma, mb;
  if (a_mn ? !make_map(&ma, A, M, K, 64, 64) : !make_map(&ma, A, K, M, 64, BM))
    return cudaErrorInvalidValue;
  if (b_mn ? !make_map(&mb, B, N, K, 64, 64) : !make_map(&mb, B, K, N, 64, 128))
    return cudaErrorInvalidValue;
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.M_host = M;
  p.N = N;
  p.Kdim = K;
  p.out = Cout;
  p.status = status;
  const int tiles = ((M + BM - 1) / BM) * ((N + 127) / 128);
  switch (layout & 3) {
    case 0: return launch_tc<128, 1, false, EPI_F32>(ma, ma, mb, mb, p, tiles, s);
    case 1: return launch_tc<128, 1, true, EPI_F32>(ma, ma, mb, mb, p, tiles, s);
    case 2: return launch_tc<128, 1, false, EPI_F32, true>(ma, ma, mb, mb, p, tiles, s);
    default: return launch_tc<128, 1, true, EPI_F32, true>(ma, ma, mb, mb, p, tiles, s);
  }
}

#endif  // TWELL_TEST_HOOKS

}  // namespace twell

#ifdef TWELL_TEST_HOOKS
extern "C" int twell_test_tc_gemm(const void *A, const void *B, float *C, int M, int N, int K,
                                  int layout, int32_t *status, void *stream) {
  if (!twell::tc_available()) return TWELL_ERR_UNSUPPORTED;
  if (!A || !B || !C || M < 1 || N < 1 || K < 8 || layout < 0 || layout > 3) return TWELL_ERR_ARG;
  if ((layout & 1) ? (N % 8) : (K % 8)) return TWELL_ERR_ARG;
  if ((layout & 2) ? (M % 8) : (K % 8)) return TWELL_ERR_ARG;
  cudaError_t e = twell::tc_test_gemm(A, B, C, M, N, K, layout, status, (cudaStream_t)stream);
  return e == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
#endif  // TWELL_TEST_HOOKS

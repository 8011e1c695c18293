// kernels.h -- host-side launchers of the TwELL kernels (internal to libtwell).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "twell.h"

namespace twell {

struct Ctl;

// Workspace carve-up shared by all entry points.
struct Workspace {
  Ctl *ctl;           // control block
  uint32_t *ovf_bits; // [ceil(T/32)] overflow-row bitmap (set by the gate epilogue)
  int32_t *rows;      // [T] rows of the dense path (hybrid: overflow rows)
  int32_t *pos;       // [T] overflow position of each row, -1 if none
  // (the row buffers hold rp rows: T, or the caller's dense-row cap, rounded
  // up to 128)
  void *h;            // [rp][F]: h rows of the dense path (bf16 gated FFN: fp16)
  void *xg;           // [rp][D] dtype: gathered x rows of the dense path (the
                      // backward's tensor-core path: fp16)
  void *wide;         // [F/C][T][C] dtype: full ReLU(z) of overflowing (tile, row)s
  void *urows;        // [Tp][F] dtype (training, CUDA-core path): u rows of the dense path
  void *dyg;          // [rp][D] (training, tensor-core path): dense-path dy rows, fp16
  void *wd16, *wg16, *wu16;  // [F][D] fp16 copies of W_down (and, training, W_gate,
                      // W_up): operands of the dense-path GEMMs (bf16 only)
  float *dbg_r;       // [Rp/32][F] fp32 (training): dbg of the dense-path rows per 32-row group
  unsigned long long *slot_parts;  // [SLOT_PARTS_MAX] per-block slot counts (backward)
  // backward scratch
  float *dz;          // [F/C][T][K] fp32: dz at the slots
  float *du;          // [F/C][T][K] fp32: du at the slots
  float *hs;          // [F/C][T][K] fp32: h at the slots (backward; the forward's two passes)
  int32_t *col_ptr;   // [F+1] neuron-major (transposed) pointers
  int32_t *col_cnt;   // [F]   per-neuron counts / cursors
  float4 *col_e;      // [T*(F/C)*K] transposed entries {token (int bits), dz, du, h}
  int32_t *col_chunk; // [(F/C) * ceil(T/1024) * C] per-(tile, token chunk) column counts
  float *dzr;         // [rp][F] fp32: dz rows of the overflow rows (gather path), or
                      // [rp][F] fp16: dz rows of the tensor-core dense-path rows
  float *dur;         // the same for du
  float *hr;          // the same for h
  int rp;             // rows of the dense-path row buffers (a multiple of 128): T
                      // rounded up, or the caller's dense-row cap rounded up
  bool dense_bufs;    // the dense-path GEMM buffers exist (the cap allows a
                      // dense-path row: cap >= T, or cap >= one 128-row tile)
  size_t bytes;       // total bytes needed
};

// Lay out (or size, when base == nullptr) the workspace; rows_cap (<= 0: T)
// bounds the rows of the dense-path buffers.
Workspace carve_workspace(void *base, int T, int D, int F, int C, int K, int dtype, int train,
                          int rows_cap);

struct FwdArgs {
  int T, D, F, C, K, dtype, gated, train;
  const void *x, *Wg, *Wu, *Wd;
  const float *bg, *rb;
  twell_t tw;
  void *y;
  Workspace ws;
  float dense_switch;
  float dense_density;  // <= 0: no density test
};

struct BwdArgs {
  int T, D, F, C, K, dtype, gated;
  const void *x, *Wg, *Wu, *Wd, *dy;
  twell_t tw;
  float lambda;
  void *dx;
  float *dWg, *dbg, *dWu, *dWd;
  Workspace ws;
  float dense_switch, dense_density;  // dispatcher of the dense-path rows (as the forward's)
  float dh_density;  // dh from a dense GEMM above this slot density (<= 0: never)
};

// Tokens per chunk of the sparse transpose (its per-(tile, chunk) column
// counts are taken where dh is finished, one per TwELL slot).
constexpr int TR_CHUNK = 1024;

// pack.cu
// Streaming multiprocessors and L2 bytes of the current device (queried once).
int num_sms();
long long l2_size();
// Passes over a gather kernel's d_model columns (or, for the forward's
// up/down, over its two matrices) so that each pass's gathered working set
// stays in L2.  requested > 0: that many (at most nv, the row's 16-byte
// vectors); 0: the fewest powers of two up to GATHER_MAX_PASSES whose share
// of set_bytes fits in GATHER_L2_SHARE of L2, keeping at least min_width
// vectors per pass.  Measured on GB300 (random
// rows, 575k gathers): 18.3 TB/s from one 34 MB matrix, 15.7 TB/s from one
// 117 MB matrix, 11.0 TB/s from two 117 MB matrices read together.  At
// d_model 4096 / d_ff 14336 (W_gate + W_up 235 MB, x + dy 134 MB at 8192
// tokens) two passes beat one (dx SpMM 1.03 -> 0.68 ms, dW 1.02 -> 0.74 ms,
// although x + dy is just below the 135.5 MB L2: the kernels also stream
// other data through it) and four (1.03, 0.84 ms: the per-pass list
// building and the narrower CTAs cost more than the smaller working set
// saves).  Column passes narrower than 256 vectors (4 KB of a bf16 row) lost
// everywhere they were measured (also d_model 2048 / 16384 tokens: dW 0.73 ->
// 0.87 ms in two passes), hence GATHER_MIN_WIDTH for the column splits.
constexpr double GATHER_L2_SHARE = 0.9;
constexpr int GATHER_MAX_PASSES = 4;
constexpr int GATHER_MIN_WIDTH = 256;
int gather_passes(int requested, double set_bytes, int nv, int min_width);

cudaError_t launch_pack_dense(const void *H, const twell_t &tw, cudaStream_t s);
// Hybrid split.  With a workspace: reads the overflow-row bitmap (which must
// hold the flags of this call), writes the row list / positions / control
// block and -- when write_user -- the caller's ovf_rows and n_ovf.  Without a
// workspace: derives the flags from nnz (one CTA) and writes only the caller's
// list and count.
// dense_density > 0: all-dense also when ctl->slots (zeroed before the gate,
// summed by its epilogue) exceeds dense_density * T * F; <= 0 ignores slots.
// slot_parts (n_parts entries, from launch_flags_from_nnz) replaces the gate
// epilogue's count in ctl->slots.  dh_density > 0 (backward): ctl->dh_gemm
// when not all-dense and the slots exceed dh_density * T * F.
// The dense path takes at most ws->rp rows (no all-dense mode when rp < T),
// none when the workspace has no dense-path buffers.
cudaError_t launch_overflow_compact(const twell_t &tw, const Workspace *ws, float dense_switch,
                                    cudaStream_t s, bool write_user = true,
                                    float dense_density = -1.f,
                                    const unsigned long long *slot_parts = nullptr,
                                    int n_parts = 0, float dh_density = -1.f);
// Overflow-row bitmap from the nnz counts (every word written); with
// slot_parts, per-block slot counts (flags_blocks(T) entries, at most
// SLOT_PARTS_MAX).
constexpr int SLOT_PARTS_MAX = 1024;
int flags_blocks(int T);
// zero (zero_n int32, may be NULL) is cleared by the same launch.
cudaError_t launch_flags_from_nnz(const twell_t &tw, uint32_t *bits,
                                  unsigned long long *slot_parts, cudaStream_t s,
                                  int32_t *zero = nullptr, long zero_n = 0);
// Dense backup rows of overflow rows that do not take the dense GEMM path.
cudaError_t launch_assemble_fb_rows(const FwdArgs &a, cudaStream_t s);
// All-dense training forward: u at the slots of the non-overflow rows.
cudaError_t launch_fill_u_slots(const FwdArgs &a, cudaStream_t s);
cudaError_t launch_copy_fb_rows(const void *H, const twell_t &tw, cudaStream_t s);
// dst[m] = src[rows[m]] for the m < n_rows overflow rows of the dense GEMM
// path (none in all-dense mode), zeros for the rows up to the next multiple
// of 128 (dst holds T rounded up to 128 rows).
cudaError_t launch_gather_rows(const void *src, void *dst, const Workspace &ws, int T, int D,
                               int dtype, cudaStream_t s);
// Backward, dense-path rows (bf16): copies the dy and x rows of the
// dense-path rows (every row in all-dense mode) into ws.dyg /
// ws.xg as fp16.
cudaError_t launch_bwd_prep_rows(const BwdArgs &a, cudaStream_t s);
// fp16 copies of up to three bf16 [F][D] matrices (src[i] -> dst[i], null
// entries skipped), done only when the dispatcher sent rows to the dense
// path (ctl->n_rows > 0); a value beyond the fp16 range records
// TWELL_ERR_RANGE.
cudaError_t launch_to_f16(const void *const src[3], void *const dst[3], size_t elems,
                          const Ctl *ctl, int32_t *status, cudaStream_t s);

// simt_gemm.cu (fp32 path)
cudaError_t launch_simt_gate_pack(const FwdArgs &a, cudaStream_t s);
cudaError_t launch_simt_dense_gu(const FwdArgs &a, cudaStream_t s);
cudaError_t launch_simt_dense_down(const FwdArgs &a, cudaStream_t s);

// tc_gemm.cu (bf16 tensor-core path)
bool tc_available();
cudaError_t launch_tc_gate_pack(const FwdArgs &a, cudaStream_t s);
cudaError_t launch_tc_dense_gu(const FwdArgs &a, cudaStream_t s);
cudaError_t launch_tc_dense_down(const FwdArgs &a, cudaStream_t s);
cudaError_t launch_tc_bwd_dh(const BwdArgs &a, cudaStream_t s);
// dh of the rows that are not on the dense path, from dy W_down^T over all
// rows, read at the TwELL slots (every CTA returns unless ctl->dh_gemm).
cudaError_t launch_tc_bwd_dh_sampled(const BwdArgs &a, cudaStream_t s);
cudaError_t launch_tc_bwd_dx(const BwdArgs &a, cudaStream_t s);
cudaError_t launch_tc_bwd_dw(const BwdArgs &a, cudaStream_t s);

// Kernel identities for the optional per-launch timing (twell_profile_*).
enum KernelId {
  KID_START = -1,
  KID_GATE_PACK = 0,
  KID_OVERFLOW_COMPACT = 1,
  KID_UPDOWN = 2,
  KID_GATHER_ROWS = 3,
  KID_DENSE_GU = 4,
  KID_DENSE_DOWN = 5,
  KID_PACK_DENSE = 6,
  KID_COPY_FB = 7,
  KID_BWD_SLOTS = 8,
  KID_BWD_DX = 9,
  KID_BWD_TRANSPOSE = 10,
  KID_BWD_DW = 11,
  KID_BWD_DENSE = 12,
  KID_FILL_U = 13,
  KID_ASSEMBLE_FB = 14,
  KID_BWD_DENSE_DX = 15,
  KID_BWD_DENSE_DW = 16,
  KID_BWD_PREP = 17,
  KID_ROWELL_PACK = 18,
  KID_ROWELL_UPDOWN = 19,
  KID_BWD_DH_GEMM = 20,
  KID_TO_F16 = 21,
  KID_COUNT = 22
};
// Record a timing event after `launches` kernel launches of component `id`
// (no-op unless enabled).
void prof_mark(int id, cudaStream_t s, int launches = 1);
// True while per-launch timing is on (the backward then stays on one stream).
bool prof_enabled();

// rowell.cu (row-ELL comparison baseline)
cudaError_t launch_rowell_pack_dense(const void *H, int T, int F, int E, int dtype, uint16_t *idx,
                                     void *val, int32_t *nnz, int32_t *status, cudaStream_t s);
cudaError_t launch_rowell_updown(const void *x, const void *Wu, const void *Wd, int T, int D,
                                 int F, int E, int dtype, const uint16_t *idx, const void *val,
                                 const int32_t *nnz, void *y, cudaStream_t s);

// updown.cu
cudaError_t launch_updown_fused(const FwdArgs &a, cudaStream_t s, int *launches = nullptr);

// backward.cu
cudaError_t launch_backward(const BwdArgs &a, cudaStream_t s);
// The library's side streams and their fork / join events, one set per host
// thread and device (created on first use, released when the thread exits):
// work forked onto s2 (or s3) after a record of `fork` (`fork3`) on the
// caller's stream is joined back by a record of `join` (`join3`) and a wait
// on the caller's stream.  `mid` orders work between the two side streams.
struct AuxStream {
  cudaStream_t s2 = nullptr, s3 = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, fork3 = nullptr, join3 = nullptr, mid = nullptr;
  AuxStream() = default;
  AuxStream(const AuxStream &) = delete;
  AuxStream &operator=(const AuxStream &) = delete;
  // (work still queued on the side streams completes; errors at process
  // teardown, when the runtime may already be unloaded, are ignored)
  ~AuxStream() {
    for (cudaEvent_t e : {mid, join3, fork3, join, fork})
      if (e) cudaEventDestroy(e);
    if (s3) cudaStreamDestroy(s3);
    if (s2) cudaStreamDestroy(s2);
  }
};
cudaError_t aux_stream(AuxStream *&out);

}  // namespace twell

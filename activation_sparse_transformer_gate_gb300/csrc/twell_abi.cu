// twell_abi.cu -- the C ABI of libtwell.so: argument checks, workspace
// carve-up and the launch sequence of each entry point (see include/twell.h).
//
// Forward launch sequence ("Sparser, Faster, Lighter Transformer Language
// Models", technical summary sections 2.A-2.B):
//   1. gate matmul + ReLU + TwELL pack epilogue         (TwELL, nnz)
//   2. overflow compaction                               (hybrid: overflow rows,
//                                                         hybrid / all-dense mode)
//   3. fused sparse up + down projection                 (non-overflow rows)
//   4. dense gate+up and down over the dense-path rows   (overflow rows, or all
//                                                         rows in all-dense mode)
// The hybrid/all-dense decision is taken on the device (step 2) and read by
// steps 3-4 from the workspace, so the host never waits for the GPU.
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace twell {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---- optional per-launch timing ---------------------------------------------
namespace {
struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> ev;
  std::vector<int> id;
  std::vector<int> nl;  // kernel launches in the interval that ends at each event
  size_t used = 0;
};
Profiler &profiler() {
  static Profiler p;
  return p;
}
}  // namespace

bool prof_enabled() { return profiler().on; }

void prof_mark(int kid, cudaStream_t s, int launches) {
  Profiler &p = profiler();
  if (!p.on) return;
  std::lock_guard<std::mutex> g(p.mu);
  if (p.used == p.ev.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return;
    p.ev.push_back(e);
    p.id.push_back(0);
    p.nl.push_back(0);
  }
  p.id[p.used] = kid;
  p.nl[p.used] = kid < 0 ? 0 : launches;
  cudaEventRecord(p.ev[p.used], s);
  ++p.used;
}

static const char *kKernelNames[KID_COUNT] = {
    "gate_gemm_relu_twell", "overflow_compact", "twell_updown_fused", "gather_rows",
    "dense_rows_gate_up",   "dense_rows_down",  "pack_dense",         "copy_fb_rows",
    "bwd_slots_sddmm",      "bwd_dx_spmm",      "twell_transpose",    "bwd_dw_gather",
    "bwd_dense_dh_gemm",    "fill_u_slots",     "assemble_fb_rows",   "bwd_dense_dx_gemm",
    "bwd_dense_dw_gemm",    "bwd_prep_rows",    "rowell_pack_dense",  "rowell_updown",
    "bwd_dh_gemm_sampled", "weights_to_f16"};

Workspace carve_workspace(void *base, int T, int D, int F, int C, int K, int dtype, int train,
                          int rows_cap) {
  Workspace w;
  memset(&w, 0, sizeof(w));
  const size_t es = dtype == TWELL_BF16 ? 2 : 4;
  const size_t nt = (size_t)F / (size_t)C;
  size_t off = 0;
  auto take = [&](size_t bytes) -> void * {
    const size_t o = off;
    off = align_up(off + (bytes ? bytes : 1), 256);
    return base ? (void *)((char *)base + o) : nullptr;
  };
  w.ctl = (Ctl *)take(sizeof(Ctl));
  w.ovf_bits = (uint32_t *)take(4 * (((size_t)T + 31) / 32));
  w.rows = (int32_t *)take(sizeof(int32_t) * (size_t)T);
  w.pos = (int32_t *)take(sizeof(int32_t) * (size_t)T);
  const size_t Tp = ((size_t)T + 127) / 128 * 128;
  // rows of the dense-path row buffers (a GEMM tile never leaves them)
  const int cap = (rows_cap <= 0 || rows_cap >= T) ? T : rows_cap;
  const size_t Rp = ((size_t)cap + 127) / 128 * 128;
  w.rp = (int)Rp;
  // Below one tile of rows (and T) no row can take the dense-path GEMMs (the
  // dispatcher sends overflow rows there from OVF_GEMM_MIN rows on): their
  // buffers are left out.
  w.dense_bufs = cap >= T || cap >= OVF_GEMM_MIN;
  auto take_dense = [&](size_t bytes) -> void * { return w.dense_bufs ? take(bytes) : nullptr; };
  w.h = take_dense(es * Rp * F);
  w.xg = take_dense(es * Rp * D);
  w.wide = take(es * Tp * F);   // indexed by token (written for overflowing tiles)
  if (dtype == TWELL_BF16) {    // fp16 operand copies of the dense-path GEMMs
    w.wd16 = take_dense(2 * (size_t)F * D);
    if (train) {
      w.wg16 = take_dense(2 * (size_t)F * D);
      w.wu16 = take_dense(2 * (size_t)F * D);
    }
  }
  const size_t slots = nt * (size_t)T * (size_t)K;
  if (!train) w.hs = (float *)take(4 * slots);  // h at the slots between the up and down passes
  if (train) {
    w.urows = take_dense(es * Rp * F);
    w.dyg = take_dense(es * Rp * D);
    w.dbg_r = (float *)take_dense(4 * (Rp / 32) * (size_t)F);
    w.slot_parts = (unsigned long long *)take(8 * (size_t)SLOT_PARTS_MAX);
    w.dz = (float *)take(4 * slots);
    w.du = (float *)take(4 * slots);
    w.hs = (float *)take(4 * slots);  // also the forward's h between its two passes
    w.col_ptr = (int32_t *)take(4 * ((size_t)F + 1));
    w.col_cnt = (int32_t *)take(4 * (size_t)F);
    w.col_e = (float4 *)take(16 * slots);
    w.col_chunk = (int32_t *)take(4 * (size_t)F * (((size_t)T + 1023) / 1024));
    // fp32 [rp][F] rows of the gather path's overflow rows, or fp16 [rp][F]
    // rows of the tensor-core backward (never both in one call)
    w.dzr = (float *)take(4 * Rp * F);
    w.dur = (float *)take(4 * Rp * F);
    w.hr = (float *)take(4 * Rp * F);
  }
  w.bytes = off;
  return w;
}

}  // namespace twell

using namespace twell;

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool pow2_k(int K) { return K == 1 || K == 2 || K == 4 || K == 8 || K == 16 || K == 32; }

twell_status check_shape(int T, int D, int F, int C, int K, int dtype) {
  if (dtype != TWELL_F32 && dtype != TWELL_BF16) return TWELL_ERR_DTYPE;
  if (T < 1 || F < 1 || D < 8) return TWELL_ERR_ARG;
  if (C != 32 && C != 64 && C != 128) return TWELL_ERR_ARG;
  if (F % C != 0 || !pow2_k(K) || K > C) return TWELL_ERR_ARG;
  const size_t es = dtype == TWELL_BF16 ? 2 : 4;
  if ((D * es) % 16 != 0 || (F * es) % 16 != 0) return TWELL_ERR_ALIGN;
  if (D * es / 16 > 1024) return TWELL_ERR_ARG;  // d_model <= 8192 (bf16) / 4096 (fp32)
  if ((double)T * (double)(F / C) * (double)K >= 2147483647.0) return TWELL_ERR_ARG;
  if ((double)T * (double)F >= 9.0e15) return TWELL_ERR_ARG;
  return TWELL_OK;
}

twell_status check_tw(const twell_t *tw, int train) {
  if (!tw) return TWELL_ERR_ARG;
  twell_status s = check_shape(tw->T, 16, tw->F, tw->C, tw->K, tw->dtype);
  if (s != TWELL_OK) return s;
  if (!tw->idx || !tw->val || !tw->nnz || !tw->n_ovf || !tw->status) return TWELL_ERR_ARG;
  if (tw->ovf_cap < 0 || tw->dense_rows_cap < 0 || tw->gather_passes < 0) return TWELL_ERR_ARG;
  if (tw->ovf_cap > 0 && (!tw->ovf_rows || !tw->g_fb)) return TWELL_ERR_ARG;
  if (!aligned16(tw->idx) || !aligned16(tw->val) || !aligned16(tw->nnz)) return TWELL_ERR_ALIGN;
  if (tw->ovf_cap > 0 && !aligned16(tw->g_fb)) return TWELL_ERR_ALIGN;
  if (train) {
    if (!tw->u_val || (tw->ovf_cap > 0 && !tw->u_fb)) return TWELL_ERR_ARG;
    if (!aligned16(tw->u_val) || (tw->ovf_cap > 0 && !aligned16(tw->u_fb))) return TWELL_ERR_ALIGN;
  }
  return TWELL_OK;
}

twell_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return TWELL_OK;
  if (e == cudaErrorNotSupported) return TWELL_ERR_UNSUPPORTED;
  return TWELL_ERR_CUDA;
}

twell_status check_ws(void *ws, size_t ws_bytes, const Workspace &need) {
  if (!ws) return TWELL_ERR_WORKSPACE;
  if (((uintptr_t)ws & 255u) != 0) return TWELL_ERR_WORKSPACE;
  if (ws_bytes < need.bytes) return TWELL_ERR_WORKSPACE;
  return TWELL_OK;
}

float switch_of(const twell_t *tw) { return tw->dense_switch > 0.f ? tw->dense_switch : 0.5f; }
// Slot density above which a call runs every row densely: the caller's
// dense_density when > 0, none when < 0, else the default crossover of the
// measured costs.  Per active (token, neuron) the forward gathers a W_up and
// a W_down row (4·d_model bytes at ~14 TB/s when those matrices sit in L2)
// where the dense path does ~4·d_model flops per (token, neuron) beyond the
// shared gate GEMM (the up and down GEMMs) at ~1.3 PFLOP/s: measured
// crossover ~1.3% at d_model 2048 / d_ff 8192.  When the gathered matrices
// exceed L2 the forward's gathers slow down even in two passes (d_model
// 4096 / d_ff 14336 bf16: 235 MB, ~13 TB/s; measured crossover ~0.9%: at
// 0.49% active 1.26 ms against 1.71 for the dense path, at 0.99% 1.76
// against 1.71), so its default is then 0.7 of the in-L2 one.  The backward gathers five rows per
// pair where its dense path does 6 GEMM units against the forward's 2 (dh,
// the two dx products, the three weight gradients): its crossover is
// (6/2) / (5/2) = 1.2 times the forward's unscaled one, with no L2 scaling:
// its dx and dW gathers run in passes whose working sets fit in L2 at close
// to the rates of the smaller shape (d_model 4096 / d_ff 14336 at 0.99%
// active: gather backward ~2.9 ms against 3.9 ms for the six GEMMs).
float density_of(const twell_t *tw, int D, int gated, bool backward) {
  if (tw->dense_density > 0.f) return tw->dense_density;
  if (tw->dense_density < 0.f) return -1.f;
  if (backward) return 0.013f * 1.2f;
  const size_t es = tw->dtype == TWELL_BF16 ? 2 : 4;
  const double wbytes = (double)(gated ? 2 : 1) * (double)tw->F * (double)D * (double)es;
  const double l2 = (double)l2_size();
  double d = 0.013;
  if (l2 > 0.0 && wbytes > l2) d *= 0.7;
  return (float)d;
}

// Slot density above which the backward takes dh from one tensor-core GEMM
// read at the slots.  Per active entry the SDDMM gathers a d_model row of
// W_down (2 d_model bytes at ~9.6 TB/s from L2); the GEMM spends 2 d_model
// flops per entry of the whole T x F product (~1.3 PFLOP/s with the
// epilogue): crossover ~0.65% (measured 0.70% at d_model 2048 / d_ff 8192,
// 0.61% at 4096 / 14336), lower when W_down does not fit in L2 and the
// gathers slow down.
float dh_density_of(const twell_t *tw, int D) {
  if (tw->dh_density > 0.f) return tw->dh_density;
  if (tw->dh_density < 0.f) return -1.f;
  const double wbytes = (double)tw->F * (double)D * (tw->dtype == TWELL_BF16 ? 2.0 : 4.0);
  const double l2 = (double)l2_size();
  double d = 0.0065;
  if (l2 > 0.0 && wbytes > l2) d *= l2 / wbytes;
  return (float)d;
}

bool use_tc(int dtype) { return dtype == TWELL_BF16 && tc_available(); }

// Steps 1-2 of the forward (shared by twell_pack and twell_ffn_forward).
cudaError_t run_gate_and_split(FwdArgs &a, cudaStream_t s) {
  // control block (its slot counter) and the overflow bitmap are adjacent
  const size_t clear = (size_t)((const char *)a.ws.ovf_bits - (const char *)a.ws.ctl) +
                       4 * (((size_t)a.T + 31) / 32);
  cudaError_t e = cudaMemsetAsync(a.ws.ctl, 0, clear, s);
  if (e != cudaSuccess) return e;
  prof_mark(KID_START, s);
  e = use_tc(a.dtype) ? launch_tc_gate_pack(a, s) : launch_simt_gate_pack(a, s);
  if (e != cudaSuccess) return e;
  prof_mark(KID_GATE_PACK, s);
  e = launch_overflow_compact(a.tw, &a.ws, a.dense_switch, s, true, a.dense_density);
  prof_mark(KID_OVERFLOW_COMPACT, s);
  return e;
}

// Step 4: dense gate+up (+ down when write_y) over the dense-path rows (none
// when the workspace has no dense-path buffers).
cudaError_t run_dense_rows(FwdArgs &a, bool write_y, cudaStream_t s) {
  if (!a.ws.dense_bufs) return cudaSuccess;
  cudaError_t e;
  if (use_tc(a.dtype)) {
    e = launch_gather_rows(a.x, a.ws.xg, a.ws, a.T, a.D, a.dtype, s);
    if (e != cudaSuccess) return e;
    prof_mark(KID_GATHER_ROWS, s);
    e = launch_tc_dense_gu(a, s);
    if (e != cudaSuccess) return e;
    prof_mark(KID_DENSE_GU, s);
    if (!write_y) return e;
    if (a.gated) {  // the down GEMM's fp16 operand copy of W_down
      const void *src[3] = {a.Wd, nullptr, nullptr};
      void *const dst[3] = {a.ws.wd16, nullptr, nullptr};
      e = launch_to_f16(src, dst, (size_t)a.F * (size_t)a.D, a.ws.ctl, a.tw.status, s);
      if (e != cudaSuccess) return e;
      prof_mark(KID_TO_F16, s);
    }
    e = launch_tc_dense_down(a, s);
    prof_mark(KID_DENSE_DOWN, s);
    return e;
  }
  e = launch_simt_dense_gu(a, s);
  if (e != cudaSuccess) return e;
  prof_mark(KID_DENSE_GU, s);
  if (!write_y) return e;
  e = launch_simt_dense_down(a, s);
  prof_mark(KID_DENSE_DOWN, s);
  return e;
}

}  // namespace

extern "C" {

const char *twell_version(void) { return "twell-gb300 0.1 (sm_103a)"; }

size_t twell_workspace_size(int T, int D, int F, int C, int K, int dtype, int train) {
  return twell_workspace_size_rows(T, D, F, C, K, dtype, train, 0);
}

size_t twell_workspace_size_rows(int T, int D, int F, int C, int K, int dtype, int train,
                                 int dense_rows_cap) {
  if (check_shape(T, D, F, C, K, dtype) != TWELL_OK) return 0;
  return carve_workspace(nullptr, T, D, F, C, K, dtype, train, dense_rows_cap).bytes;
}

twell_status twell_pack_dense(const void *H, twell_t *tw, void *stream) {
  twell_status st = check_tw(tw, 0);
  if (st != TWELL_OK) return st;
  if (!H) return TWELL_ERR_ARG;
  if (!aligned16(H)) return TWELL_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  prof_mark(KID_START, s);
  cudaError_t e = launch_pack_dense(H, *tw, s);
  prof_mark(KID_PACK_DENSE, s);
  if (e == cudaSuccess) e = launch_overflow_compact(*tw, nullptr, 1.0f, s);
  prof_mark(KID_OVERFLOW_COMPACT, s);
  if (e == cudaSuccess) e = launch_copy_fb_rows(H, *tw, s);
  prof_mark(KID_COPY_FB, s);
  return cuda_status(e);
}

twell_status twell_pack(const void *x, const void *Wg, const float *bg, const float *row_bias,
                        int D, twell_t *tw, void *workspace, size_t workspace_bytes,
                        void *stream) {
  twell_status st = check_tw(tw, 0);
  if (st != TWELL_OK) return st;
  st = check_shape(tw->T, D, tw->F, tw->C, tw->K, tw->dtype);
  if (st != TWELL_OK) return st;
  if (!x || !Wg || !bg) return TWELL_ERR_ARG;
  if (!aligned16(x) || !aligned16(Wg)) return TWELL_ERR_ALIGN;
  Workspace need = carve_workspace(nullptr, tw->T, D, tw->F, tw->C, tw->K, tw->dtype, 0, tw->dense_rows_cap);
  st = check_ws(workspace, workspace_bytes, need);
  if (st != TWELL_OK) return st;
  FwdArgs a;
  memset(&a, 0, sizeof(a));
  a.T = tw->T; a.D = D; a.F = tw->F; a.C = tw->C; a.K = tw->K; a.dtype = tw->dtype;
  a.gated = 0; a.train = 0; a.x = x; a.Wg = Wg; a.bg = bg; a.rb = row_bias; a.tw = *tw;
  a.ws = carve_workspace(workspace, a.T, D, a.F, a.C, a.K, a.dtype, 0, tw->dense_rows_cap);
  a.dense_switch = 2.0f;  // the pack never switches to all-dense mode
  a.dense_density = -1.f;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = run_gate_and_split(a, s);
  if (e == cudaSuccess) {  // dense backup rows: assembled (few rows) or recomputed (many)
    e = launch_assemble_fb_rows(a, s);
    prof_mark(KID_ASSEMBLE_FB, s);
  }
  if (e == cudaSuccess) e = run_dense_rows(a, false, s);
  return cuda_status(e);
}

twell_status twell_ffn_forward(const void *x, const void *Wg, const float *bg,
                               const float *row_bias, const void *Wu, const void *Wd, int D,
                               int train, twell_t *tw, void *y, void *workspace,
                               size_t workspace_bytes, void *stream) {
  const int gated = Wu != nullptr;
  twell_status st = check_tw(tw, train && gated);
  if (st != TWELL_OK) return st;
  st = check_shape(tw->T, D, tw->F, tw->C, tw->K, tw->dtype);
  if (st != TWELL_OK) return st;
  if (!x || !Wg || !bg || !Wd || !y) return TWELL_ERR_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wd) || !aligned16(y) ||
      (Wu && !aligned16(Wu)))
    return TWELL_ERR_ALIGN;
  Workspace need = carve_workspace(nullptr, tw->T, D, tw->F, tw->C, tw->K, tw->dtype, train, tw->dense_rows_cap);
  st = check_ws(workspace, workspace_bytes, need);
  if (st != TWELL_OK) return st;
  FwdArgs a;
  memset(&a, 0, sizeof(a));
  a.T = tw->T; a.D = D; a.F = tw->F; a.C = tw->C; a.K = tw->K; a.dtype = tw->dtype;
  a.gated = gated; a.train = train ? 1 : 0;
  a.x = x; a.Wg = Wg; a.Wu = Wu; a.Wd = Wd; a.bg = bg; a.rb = row_bias; a.tw = *tw; a.y = y;
  a.ws = carve_workspace(workspace, a.T, D, a.F, a.C, a.K, a.dtype, train, tw->dense_rows_cap);
  a.dense_switch = switch_of(tw);
  a.dense_density = density_of(tw, D, gated, false);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = run_gate_and_split(a, s);
  // The dense-path rows (tensor cores) and the gathers own disjoint rows:
  // the dense-path kernels run on the library's second stream, launched
  // first, beside the up/down gathers (one stream while per-launch timing
  // is on).  With few dense-path rows their GEMMs fill a fraction of the
  // GPU for a whole wave, which the gathers then use.
  const bool fork = e == cudaSuccess && use_tc(a.dtype) && !prof_enabled();
  AuxStream *aux = nullptr;
  if (fork) {
    e = aux_stream(aux);
    if (e == cudaSuccess) e = cudaEventRecord(aux->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(aux->s2, aux->fork, 0);
    if (e != cudaSuccess) return cuda_status(e);
    e = run_dense_rows(a, true, aux->s2);
  }
  if (e == cudaSuccess) {
    int n = 1;
    e = launch_updown_fused(a, s, &n);
    prof_mark(KID_UPDOWN, s, n);
  }
  if (fork) {  // join (also after an error, so the caller's stream stays ordered)
    const cudaError_t j1 = cudaEventRecord(aux->join, aux->s2);
    const cudaError_t j2 = j1 == cudaSuccess ? cudaStreamWaitEvent(s, aux->join, 0) : j1;
    if (e == cudaSuccess) e = j2;
  } else if (e == cudaSuccess) {
    e = run_dense_rows(a, true, s);
  }
  // all-dense training: u at the slots of non-overflow rows (the tensor-core
  // up GEMM writes them in its epilogue)
  if (e == cudaSuccess && a.train && a.gated && !use_tc(a.dtype) && a.ws.dense_bufs) {
    e = launch_fill_u_slots(a, s);
    prof_mark(KID_FILL_U, s);
  }
  return cuda_status(e);
}

twell_status twell_ffn_backward(const void *x, const void *Wg, const void *Wu, const void *Wd,
                                const twell_t *tw, const void *dy, float lambda, int D,
                                void *dx, float *dWg, float *dbg, float *dWu, float *dWd,
                                void *workspace, size_t workspace_bytes, void *stream) {
  const int gated = Wu != nullptr;
  twell_status st = check_tw(tw, gated);
  if (st != TWELL_OK) return st;
  st = check_shape(tw->T, D, tw->F, tw->C, tw->K, tw->dtype);
  if (st != TWELL_OK) return st;
  if (!x || !Wg || !Wd || !dy || !dx || !dWg || !dbg || !dWd || (gated && !dWu))
    return TWELL_ERR_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wd) || !aligned16(dy) || !aligned16(dx) ||
      !aligned16(dWg) || !aligned16(dWd) || (gated && (!aligned16(Wu) || !aligned16(dWu))))
    return TWELL_ERR_ALIGN;
  Workspace need = carve_workspace(nullptr, tw->T, D, tw->F, tw->C, tw->K, tw->dtype, 1, tw->dense_rows_cap);
  st = check_ws(workspace, workspace_bytes, need);
  if (st != TWELL_OK) return st;
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.T = tw->T; a.D = D; a.F = tw->F; a.C = tw->C; a.K = tw->K; a.dtype = tw->dtype;
  a.gated = gated; a.x = x; a.Wg = Wg; a.Wu = Wu; a.Wd = Wd; a.dy = dy; a.tw = *tw;
  a.lambda = lambda; a.dx = dx; a.dWg = dWg; a.dbg = dbg; a.dWu = dWu; a.dWd = dWd;
  a.dense_switch = switch_of(tw);
  a.dense_density = density_of(tw, D, gated, true);
  a.dh_density = dh_density_of(tw, D);
  a.ws = carve_workspace(workspace, a.T, D, a.F, a.C, a.K, a.dtype, 1, tw->dense_rows_cap);
  // the backward keeps the gradients of an overflow row on the gather path in
  // the workspace's row buffers: at most rp of them
  if (a.tw.ovf_cap > a.ws.rp) a.tw.ovf_cap = a.ws.rp;
  return cuda_status(launch_backward(a, (cudaStream_t)stream));
}

static twell_status check_rowell(const twell_rowell_t *re) {
  if (!re) return TWELL_ERR_ARG;
  if (re->dtype != TWELL_F32 && re->dtype != TWELL_BF16) return TWELL_ERR_DTYPE;
  if (re->T < 1 || re->F < 32 || re->F % 32 != 0 || re->F > 65535 || re->E < 1)
    return TWELL_ERR_ARG;
  if ((double)re->T * (double)re->E >= 2147483647.0) return TWELL_ERR_ARG;
  if (!re->idx || !re->val || !re->nnz || !re->status) return TWELL_ERR_ARG;
  if (!aligned16(re->val)) return TWELL_ERR_ALIGN;
  return TWELL_OK;
}

twell_status twell_rowell_pack_dense(const void *H, twell_rowell_t *re, void *stream) {
  twell_status st = check_rowell(re);
  if (st != TWELL_OK) return st;
  if (!H) return TWELL_ERR_ARG;
  if (!aligned16(H)) return TWELL_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  prof_mark(KID_START, s);
  cudaError_t e = launch_rowell_pack_dense(H, re->T, re->F, re->E, re->dtype, re->idx, re->val,
                                           re->nnz, re->status, s);
  prof_mark(KID_ROWELL_PACK, s);
  return cuda_status(e);
}

twell_status twell_rowell_forward(const void *x, const void *Wu, const void *Wd, int D,
                                  const twell_rowell_t *re, void *y, void *stream) {
  twell_status st = check_rowell(re);
  if (st != TWELL_OK) return st;
  if (!x || !Wd || !y) return TWELL_ERR_ARG;
  const size_t es = re->dtype == TWELL_BF16 ? 2 : 4;
  if (D < 8 || (D * es) % 16 != 0 || D * es > 16384) return D < 8 ? TWELL_ERR_ARG : TWELL_ERR_ALIGN;
  if (!aligned16(x) || !aligned16(Wd) || !aligned16(y) || (Wu && !aligned16(Wu)))
    return TWELL_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  prof_mark(KID_START, s);
  cudaError_t e = launch_rowell_updown(x, Wu, Wd, re->T, D, re->F, re->E, re->dtype, re->idx,
                                       re->val, re->nnz, y, s);
  prof_mark(KID_ROWELL_UPDOWN, s);
  return cuda_status(e);
}

int twell_profile_begin(void) {
  Profiler &p = profiler();
  std::lock_guard<std::mutex> g(p.mu);
  p.used = 0;
  p.on = true;
  return TWELL_OK;
}

int twell_profile_end(int capacity, int *kernel_ids, float *ms, int *count) {
  return twell_profile_end_ex(capacity, kernel_ids, ms, nullptr, count);
}

int twell_profile_end_ex(int capacity, int *kernel_ids, float *ms, int *launches, int *count) {
  Profiler &p = profiler();
  std::lock_guard<std::mutex> g(p.mu);
  p.on = false;
  int n = 0;
  for (size_t i = 1; i < p.used; ++i) {
    if (p.id[i] < 0) continue;  // an entry point's start marker
    if (cudaEventSynchronize(p.ev[i]) != cudaSuccess) return TWELL_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, p.ev[i - 1], p.ev[i]) != cudaSuccess) return TWELL_ERR_CUDA;
    if (n < capacity) {
      if (kernel_ids) kernel_ids[n] = p.id[i];
      if (ms) ms[n] = t;
      if (launches) launches[n] = p.nl[i];
    }
    ++n;
  }
  if (count) *count = n;
  p.used = 0;
  return n <= capacity ? TWELL_OK : TWELL_ERR_CAPACITY;
}

const char *twell_kernel_name(int kernel_id) {
  return (kernel_id >= 0 && kernel_id < KID_COUNT) ? kKernelNames[kernel_id] : "unknown";
}

twell_status twell_get_status(const twell_t *tw, void *stream, int32_t *n_ovf) {
  if (!tw || !tw->status) return TWELL_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t host[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(&host[0], tw->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && n_ovf && tw->n_ovf)
    e = cudaMemcpyAsync(&host[1], tw->n_ovf, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(tw->status, 0, sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return TWELL_ERR_CUDA;
  if (n_ovf) *n_ovf = host[1];
  return (twell_status)host[0];
}

}  // extern "C"

/*
 * twell.h -- C ABI of libtwell.so: the activation-sparse transformer FFN with
 * the Tile-wise ELLPACK (TwELL) format, for one GB300 (sm_103a).
 *
 * Source: "Sparser, Faster, Lighter Transformer Language Models" (Cetin,
 * Peluchetti, Castillo, Naruse, Murakami, Jones; arXiv 2603.23198), as
 * explained on gist.science, technical summary:
 *   section 2.A  TwELL: the columns of the hidden activation matrix are cut into
 *                tiles; each (row, tile) keeps a fixed number K of (index,
 *                value) slots, produced directly in the epilogue of the dense
 *                gate matmul without inter-CTA synchronisation.
 *   section 2.A  hybrid format: rows whose non-zeros do not fit go to a dense
 *                backup matrix ("overflow").
 *   section 2.B  inference: one fused kernel does the up and down projections
 *                from the TwELL gate activations; training: TwELL -> hybrid,
 *                hybrid x dense and dense x hybrid products, sparse transposes.
 *   section 2.B  L1 regularisation of the ReLU FFN activations.
 *
 * The FFN (gated):  z = x Wg^T + bg (+ row_bias), g = ReLU(z), u = x Wu^T,
 *                   h = g * u, y = h Wd.   Plain (Wu == NULL): h = g.
 *
 * Shapes (T tokens, D = d_model, F = d_ff, C = tile width, K = slots):
 *   x, y, dy, dx         [T][D]  row-major, element type `dtype`
 *   Wg, Wu               [F][D]  row-major (row n = neuron n; nn.Linear layout)
 *   Wd                   [F][D]  row-major NEURON-MAJOR: the transpose of the
 *                                nn.Linear [D][F] down weight, so that the
 *                                row of an active neuron is contiguous
 *   bg [F], row_bias [T] fp32 (row_bias may be NULL)
 *   dWg, dWu, dWd        [F][D]  fp32, dbg [F] fp32
 *
 * TwELL layout (tile-major):  tile j covers hidden columns [j*C, (j+1)*C).
 *   idx [F/C][T][K]  uint8, local column of the slot, ascending; pad 0xFF
 *   val [F/C][T][K]  dtype, ReLU(z) rounded to dtype (RNE); pad +0
 *   nnz [F/C][T]     uint8, TRUE number of positive z in (row, tile); may be > K
 *   A row is an overflow row iff some tile has nnz > K.  Its slots are still
 *   written (first K ascending), and its full ReLU(z) row goes to the dense
 *   backup g_fb; overflow rows are listed in ascending order in ovf_rows.
 *   A value is active iff z > 0 in fp32 (ReLU(0) = 0).
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers, owned by the caller; the library
 *     never allocates or keeps device memory.  Scratch comes from the caller's
 *     `workspace` of at least twell_workspace_size(...) bytes (256-byte
 *     aligned).
 *   - All calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Errors the host can see (shape, dtype, NULL, alignment,
 *     workspace size) are returned before anything is launched.  Errors that
 *     only the device can see are written to *tw->status (first error wins)
 *     and are read by twell_get_status; after such an error the outputs are
 *     undefined.
 *   - Alignment: every pointer 16-byte aligned; D*elem_size and F*elem_size
 *     multiples of 16 bytes.
 *   - Supported: dtype F32 (CUDA-core FFMA, no TF32) and BF16 (tensor cores,
 *     fp32 accumulation); C in {32, 64, 128}; F % C == 0;
 *     K in {1, 2, 4, 8, 16, 32}, K <= C; 1 <= T; 8 <= D with
 *     D*elem_size <= 16384 bytes (d_model <= 8192 in bf16, <= 4096 in fp32);
 *     T*(F/C)*K < 2^31.  Other shapes return TWELL_ERR_ARG.
 *   - Thread safety: calls on distinct twell_t / workspaces may run
 *     concurrently on different streams.
 */
#ifndef TWELL_H
#define TWELL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TWELL_OK = 0,
  TWELL_ERR_ARG = -1,        /* bad shape, NULL pointer, unsupported C/K     */
  TWELL_ERR_ALIGN = -2,      /* pointer or row pitch not 16-byte aligned     */
  TWELL_ERR_DTYPE = -3,      /* unknown dtype                                */
  TWELL_ERR_CAPACITY = -4,   /* device: more overflow rows than ovf_cap      */
  TWELL_ERR_INDEX = -5,      /* device: malformed TwELL (slot index >= C)    */
  TWELL_ERR_TIMEOUT = -6,    /* device: a bounded pipeline wait expired      */
  TWELL_ERR_CUDA = -7,       /* a CUDA runtime/driver call failed            */
  TWELL_ERR_WORKSPACE = -8,  /* workspace NULL, misaligned or too small      */
  TWELL_ERR_UNSUPPORTED = -9,/* valid request this build does not implement  */
  TWELL_ERR_STATIC_LIMIT = -10,/* size above a fixed static-scratch maximum   */
  TWELL_ERR_RANGE = -11      /* device: a dense-path value beyond the fp16
                                range (|v| > 65504) of the tensor-core
                                operands of the dense-path rows            */
} twell_status;

typedef enum { TWELL_F32 = 0, TWELL_BF16 = 1 } twell_dtype;

/* TwELL + hybrid activations of one FFN call.  All pointers: device memory,
 * caller-owned.  Filled by twell_pack / twell_ffn_forward, read by
 * twell_ffn_backward. */
typedef struct {
  int32_t T, F, C, K;     /* tokens, hidden width, tile width, slots/tile   */
  int32_t dtype;          /* twell_dtype of val, g_fb, u_val, u_fb          */
  uint8_t *idx;           /* [F/C][T][K]                                     */
  void *val;              /* [F/C][T][K]                                     */
  uint8_t *nnz;           /* [F/C][T]                                        */
  int32_t *ovf_rows;      /* [ovf_cap] ascending overflow rows               */
  int32_t *n_ovf;         /* device scalar: true number of overflow rows     */
  int32_t ovf_cap;        /* rows that ovf_rows / g_fb / u_fb can hold (>= 0)*/
  void *g_fb;             /* [ovf_cap][F] dense ReLU(z) rows (dense backup)  */
  void *u_val;            /* training: [F/C][T][K] u = x.Wu[n] at the slots  */
  void *u_fb;             /* training: [ovf_cap][F] u rows of overflow rows  */
  int32_t *status;        /* device int32, must be 0 before the first call   */
  float dense_switch;     /* forward runs every row densely when
                             n_ovf > dense_switch * T; <= 0 selects 0.5      */
  float dense_density;    /* ... or when the slots written (active entries,
                             at most K per row and tile) exceed
                             dense_density * T * F: at such densities the
                             gathers cost more than dense GEMMs.  0 selects
                             the measured crossover: in the forward 0.013
                             when the gathered weights (W_up + W_down) fit
                             in L2, 0.0091 when they do not; in the backward
                             0.0156 (its gathers run in L2-sized passes);
                             < 0 disables this test.
                             The backward applies the same rules to the
                             saved TwELL.                                    */
  float dh_density;       /* backward, bf16 on the tensor-core path: when the
                             rows are not all dense and the slots exceed
                             dh_density * T * F, dh of the rows the gathers
                             own comes from one dense GEMM dy W_down^T read
                             at the slots instead of the per-entry SDDMM
                             (same values up to fp32 summation order).  0
                             selects the measured crossover: 0.0065, scaled
                             by L2 / bytes of W_down when W_down does not fit
                             in L2; < 0 always gathers.                      */
  int32_t dense_rows_cap; /* rows the workspace's dense-path buffers hold
                             (0: T).  With a cap R < T the workspace is sized
                             by twell_workspace_size_rows(..., R): the
                             dispatcher then never runs more than R rows on
                             the dense path (no all-dense mode; overflow rows
                             beyond R stay on the gathers), and the backward
                             keeps the gradients of at most min(ovf_cap, R)
                             overflow rows (more: TWELL_ERR_CAPACITY).  The
                             same value must be used for the workspace size
                             and every call.                                 */
  int32_t gather_passes;  /* passes of the row-gather kernels over their
                             gathered matrices, so that each pass's working
                             set stays in L2: the forward's up and down
                             projections run as one pass or as an up pass
                             then a down pass (gated FFN, >= 2); the
                             backward's dx and weight-gradient gathers split
                             d_model into this many column ranges, and the
                             weight gradients also gather x rows (dW_gate,
                             dW_up, dbg) and dy rows (dW_down) in separate
                             launches (>= 2).  Results are bit-identical for
                             every value.  0 selects it from the working set
                             (W_up + W_down; W_gate + W_up; x + dy) against
                             the L2 size; >= 1 forces it (the column split
                             at most d_model / 8 (bf16) or d_model / 4
                             (fp32) passes).                                 */
} twell_t;

/* Bytes of scratch that twell_pack / twell_ffn_forward / twell_ffn_backward
 * need for these sizes (train != 0: forward with saved activations and the
 * backward).  Returns 0 for invalid sizes. */
size_t twell_workspace_size(int T, int D, int F, int C, int K, int dtype, int train);

/* The same with the dense-path row buffers sized for dense_rows_cap rows
 * (<= 0 or >= T: T rows, as twell_workspace_size).  A cap trades the
 * all-dense fallback for memory: the dense-path buffers are the bulk of the
 * workspace (with training, ~13 bytes x d_ff per row, plus the d_model rows). */
size_t twell_workspace_size_rows(int T, int D, int F, int C, int K, int dtype, int train,
                                 int dense_rows_cap);

/* Pack a dense post-ReLU activation matrix H [T][F] (dtype = tw->dtype, all
 * entries >= 0) into TwELL + hybrid (section 2.A).  Fills idx, val, nnz,
 * ovf_rows, n_ovf, g_fb (first min(n_ovf, ovf_cap) rows; CAPACITY is raised
 * on the device when n_ovf > ovf_cap).  Entries > 0 are active. */
twell_status twell_pack_dense(const void *H, twell_t *tw, void *stream);

/* Gate matmul with the ReLU + TwELL-packing epilogue (section 2.A):
 * z = x Wg^T + bg (+ row_bias), then the TwELL slots, nnz, the overflow row
 * list and the dense backup rows g_fb of the overflow rows. */
twell_status twell_pack(const void *x, const void *Wg, const float *bg, const float *row_bias,
                        int D, twell_t *tw, void *workspace, size_t workspace_bytes,
                        void *stream);

/* FFN forward (sections 2.A + 2.B): twell_pack, then the fused up + down
 * projection over the TwELL slots for non-overflow rows, and dense up + down
 * for the overflow rows (all rows when n_ovf > dense_switch * T or the
 * slots exceed dense_density * T * F).
 * Wu == NULL selects the plain FFN y = ReLU(z) Wd.  y [T][D] dtype.
 * train != 0 additionally stores u at the slots (tw->u_val) and the u rows of
 * the overflow rows (tw->u_fb) for twell_ffn_backward.
 * Ordering: on the bf16 tensor-core path the dense-row kernels run on the
 * library's second stream (as in twell_ffn_backward), forked from `stream`
 * after the overflow split and joined back before the call returns. */
twell_status twell_ffn_forward(const void *x, const void *Wg, const float *bg,
                               const float *row_bias, const void *Wu, const void *Wd, int D,
                               int train, twell_t *tw, void *y, void *workspace,
                               size_t workspace_bytes, void *stream);

/* FFN backward with the L1 term lambda * sum |h| (section 2.B), from the
 * activations a training forward left in *tw (same x, weights, row_bias):
 *   dh = dy . Wd[n] + lambda sign(h);  dz = [z>0] dh u;  du = dh g
 *   dx = sum_n dz Wg[n] + du Wu[n]     (dtype)
 *   dWg[n] = sum_t dz x_t, dbg[n] = sum_t dz, dWu[n] = sum_t du x_t,
 *   dWd[n] = sum_t h dy_t              (fp32, overwritten, not accumulated)
 * Plain FFN (Wu == NULL, dWu ignored): dz = [z>0] dh.  Only active (row,
 * neuron) pairs are visited; rows of never-active neurons are written 0.
 * Ordering: the weight-gradient kernels run on a second stream of the
 * library (one per host thread and device, created on first use), forked
 * from `stream` after dh and joined back with events before the call
 * returns, so all work is ordered with `stream` as if it ran there (also
 * under stream capture).  While per-launch timing (twell_profile_begin) is
 * on, everything runs on `stream`. */
twell_status twell_ffn_backward(const void *x, const void *Wg, const void *Wu, const void *Wd,
                                const twell_t *tw, const void *dy, float lambda, int D,
                                void *dx, float *dWg, float *dbg, float *dWu, float *dWd,
                                void *workspace, size_t workspace_bytes, void *stream);

/* Synchronise `stream`, read the device status word of *tw (and, if n_ovf is
 * not NULL, the overflow-row count), then clear the status word.  Returns the
 * device status (TWELL_OK when no error was recorded) or TWELL_ERR_CUDA. */
twell_status twell_get_status(const twell_t *tw, void *stream, int32_t *n_ovf);

/* Overflow-row list of an already packed TwELL, for callers that cannot
 * allocate device memory (the paper has no counterpart: this is a library
 * convenience).  Such callers -- code running inside an allocator or memory
 * pool it does not own, plugin hosts that forbid allocation on their hot
 * path -- cannot provide the workspace the other entry points take.  This
 * call reads tw->nnz and writes tw->ovf_rows (first min(n, ovf_cap) rows,
 * ascending), *tw->n_ovf and, when n > ovf_cap, TWELL_ERR_CAPACITY to the
 * status word; it does not touch g_fb.  Its scratch is a fixed device array
 * inside the library (about 2 MiB, held on every GPU that loads the library
 * until the process exits), so it allocates nothing.
 *   - T > TWELL_STATIC_SPLIT_MAX_T returns TWELL_ERR_STATIC_LIMIT before any
 *     launch.
 *   - The first call in each CUDA context (each device's primary context, and
 *     again after a device reset) looks the array's address up with that
 *     context current; make that first call before any stream capture.
 *   - All calls share the array: calls that overlap on the GPU race.  The
 *     array keeps the last call's contents; each call clears what it needs. */
#define TWELL_STATIC_SPLIT_MAX_T 262144
twell_status twell_hybrid_split_static(twell_t *tw, void *stream);

/* Comparison baseline (not on the TwELL path): classic row-ELL, the format
 * the technical summary (section 2.A) contrasts TwELL with.  One list per
 * row over the whole hidden axis, padded to a common width E:
 *   idx [T][E]  uint16 global hidden column, ascending; pad 0xFFFF
 *   val [T][E]  dtype, the activation value; pad +0
 *   nnz [T]     int32, the row's TRUE number of positive values
 * A row spans every N-tile of the gate matmul, so row-ELL cannot be written
 * in its epilogue: it is packed from a dense activation matrix by a separate
 * pass.  Rows with more than E positive values keep their first E (nnz stays
 * true) and TWELL_ERR_CAPACITY goes to *status; a caller who wants no loss
 * picks E = the densest row's count.  F <= 65535. */
typedef struct {
  int32_t T, F, E;        /* tokens, hidden width, entries per row          */
  int32_t dtype;          /* twell_dtype of val                              */
  uint16_t *idx;          /* [T][E]                                          */
  void *val;              /* [T][E]                                          */
  int32_t *nnz;           /* [T]                                             */
  int32_t *status;        /* device int32 (first error wins)                 */
} twell_rowell_t;

/* Pack a dense activation matrix H [T][F] (dtype = re->dtype, entries >= 0;
 * entries > 0 are active) into row-ELL. */
twell_status twell_rowell_pack_dense(const void *H, twell_rowell_t *re, void *stream);

/* y [T][D] = sum over each row's entries of h W_down[n], with h = g u,
 * u = x . W_up[n] (gated), or h = g (Wu == NULL): the up + down projection
 * of the FFN consuming row-ELL gate activations.  x, Wu, Wd, y as for
 * twell_ffn_forward; D*elem_size <= 16384 bytes. */
twell_status twell_rowell_forward(const void *x, const void *Wu, const void *Wd, int D,
                                  const twell_rowell_t *re, void *y, void *stream);

/* Optional per-launch timing, for benchmarks.  Between twell_profile_begin
 * and twell_profile_end every entry point records a CUDA event on its stream
 * before its first kernel and after each step of its launch sequence (a step
 * is one kernel, or a few launches of one component: the overflow-row flags
 * and their scan, the backward's dense-path row gathers).  twell_profile_end
 * waits for those events and returns, in launch order, the step's identity
 * (see twell_kernel_name) and the milliseconds between the event before and
 * the event after it; *count receives the number of steps
 * (TWELL_ERR_CAPACITY when it exceeds `capacity`).  twell_profile_end_ex
 * also returns the kernel launches of each step (launches may be NULL).
 * Recording is process-wide; the events are created once and reused. */
int twell_profile_begin(void);
int twell_profile_end(int capacity, int *kernel_ids, float *ms, int *count);
int twell_profile_end_ex(int capacity, int *kernel_ids, float *ms, int *launches, int *count);
const char *twell_kernel_name(int kernel_id);

/* Version string of the library build. */
const char *twell_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TWELL_H */

/*
 * twell_oracle.c -- CPU oracle for the activation-sparse FFN and its TwELL
 * packing.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the CUDA library never does, and the
 * two share no code.
 *
 * Source ("Sparser, Faster, Lighter Transformer Language Models",
 * gist.science explainer, technical summary):
 *   section 2.A  TwELL: the columns of the activation matrix are cut into
 *                tiles and each (row, tile) keeps a fixed number of
 *                (index, value) slots; the format is produced in the epilogue
 *                of the dense gate matmul.
 *   section 2.A  hybrid format: rows whose non-zeros do not fit the compact
 *                ELL part go to a dense backup matrix.
 *   section 2.B  inference: up and down projections consume the gate
 *                activations stored in TwELL; training: hybrid-dense and
 *                dense-hybrid products and sparse transposes for gradients.
 *   section 2.B  L1 penalty on the ReLU FFN activations.
 *   section 5    the only model change is the ReLU activation + the L1 term.
 *
 * Readings of what the pages leave open (each is a choice, listed with its
 * reason in the design notes):
 *   - tiles are contiguous C-column ranges of the hidden (d_ff) axis;
 *   - a slot holds the column index local to its tile and the gate value;
 *     slots are filled in ascending column order, unused slots hold index
 *     0xFF and value +0;
 *   - nnz keeps the true count of the (row, tile) even when it exceeds K;
 *   - a row is an overflow row iff any of its tiles has more than K
 *     non-zeros; its full ReLU(gate) row goes to the dense backup matrix,
 *     overflow rows listed in ascending order;
 *   - active <=> z > 0 strictly (ReLU(0) = 0);
 *   - gated FFN: h = ReLU(z) * u, u = x . W_up[n]; y = sum_n h W_down[n];
 *     plain FFN: h = ReLU(z); W_down is stored neuron-major [F][D];
 *   - L1 term lambda * sum |h| with sign(0) = 0 and no 1/T factor.
 *
 * Arithmetic: every sum is a plain loop in ascending index order, in double
 * precision.  Inputs (fp32 or bf16) widen exactly.  Where a floating-point
 * value decides an integer (is z > 0?), the decision is taken on z rounded to
 * fp32, the precision in which the GPU kernel takes it.  Values that the
 * format stores (TwELL values, dense backup rows) are rounded to the storage
 * type (fp32 or bf16, round-to-nearest-even) and the forward/backward consume
 * those rounded gate values, exactly as the format delivers them.  A third
 * rounding mode (none) keeps everything in double precision; it serves the
 * finite-difference pins.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC.  OpenMP only
 * splits independent rows (tokens for forward / dx, neurons for dW), so the
 * results do not depend on the number of threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1 };            /* storage type of x, W, dy      */
enum { Q_F32 = 0, Q_BF16 = 1, Q_NONE = 2 };  /* rounding of stored activations */

/* ---- scalar helpers ---------------------------------------------------- */

static double ld(const void *p, int dt, size_t i) {
  if (dt == OR_BF16) {
    uint32_t b = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
  }
  return (double)((const float *)p)[i];
}

/* float -> bfloat16 bit pattern, round to nearest, ties to even (finite). */
static uint16_t bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Storage rounding of an activation value. */
static double quant(double v, int q) {
  if (q == Q_NONE) return v;
  float f = (float)v;
  if (q == Q_F32) return (double)f;
  return bf16_value(bf16_bits(f));
}

/* The activity decision: z > 0, taken in fp32 unless q == Q_NONE. */
static int is_active(double z, int q) {
  if (q == Q_NONE) return z > 0.0;
  return (float)z > 0.0f;
}

static double sgn(double v) { return v > 0.0 ? 1.0 : (v < 0.0 ? -1.0 : 0.0); }

/* dot(a[ia..], b[ib..]) over D elements, ascending. */
static double dot(const void *a, int dta, size_t ia, const void *b, int dtb, size_t ib, int D) {
  double s = 0.0;
  for (int d = 0; d < D; ++d) s += ld(a, dta, ia + (size_t)d) * ld(b, dtb, ib + (size_t)d);
  return s;
}

/* ---- public entry points ----------------------------------------------- */

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Round fp32 values to bf16 bit patterns (exposed so that the rounding can be
 * pinned against independent implementations). */
void oracle_bf16_round(const float *in, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits(in[i]);
}

/* Gate pre-activation (section 2.A: the dense gate matmul that TwELL is
 * produced from):  z[t][n] = sum_d x[t][d] * Wg[n][d] + bg[n] + rb[t].
 * x [T][D], Wg [F][D] in storage type dt; bg [F] fp32; rb [T] fp32 or NULL. */
void oracle_gate(int T, int D, int F, int dt, const void *x, const void *Wg,
                 const float *bg, const float *rb, double *z) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int n = 0; n < F; ++n) {
      double s = dot(x, dt, (size_t)t * D, Wg, dt, (size_t)n * D, D);
      s += (double)bg[n];
      if (rb) s += (double)rb[t];
      z[(size_t)t * F + n] = s;
    }
  }
}

/* TwELL pack + hybrid split (section 2.A).
 * Outputs: idx [nt][T][K] (local column, 0xFF pad), val [nt][T][K] (stored,
 * rounded value, +0 pad), nnz [nt][T] (true count), row_ovf [T] (0/1),
 * ovf_rows [T] (ascending overflow rows), g_fb [T][F] (rows 0..n_ovf-1:
 * full rounded ReLU rows of the overflow rows).  Returns n_ovf. */
int oracle_twell_pack(int T, int F, int C, int K, int q, const double *z,
                      uint8_t *idx, double *val, uint8_t *nnz, uint8_t *row_ovf,
                      int32_t *ovf_rows, double *g_fb) {
  int nt = F / C;
  for (int t = 0; t < T; ++t) {
    int over = 0;
    for (int j = 0; j < nt; ++j) {
      size_t s0 = ((size_t)j * T + t) * (size_t)K;
      for (int k = 0; k < K; ++k) {
        idx[s0 + k] = 0xFF;
        val[s0 + k] = 0.0;
      }
      int cnt = 0;
      for (int c = 0; c < C; ++c) {
        double zz = z[(size_t)t * F + (size_t)j * C + c];
        if (!is_active(zz, q)) continue;
        if (cnt < K) {
          idx[s0 + cnt] = (uint8_t)c;
          val[s0 + cnt] = quant(zz, q);
        }
        ++cnt;
      }
      nnz[(size_t)j * T + t] = (uint8_t)cnt;
      if (cnt > K) over = 1;
    }
    row_ovf[t] = (uint8_t)over;
  }
  int n_ovf = 0;
  for (int t = 0; t < T; ++t) {
    if (!row_ovf[t]) continue;
    ovf_rows[n_ovf] = t;
    for (int n = 0; n < F; ++n) {
      double zz = z[(size_t)t * F + n];
      g_fb[(size_t)n_ovf * F + n] = is_active(zz, q) ? quant(zz, q) : 0.0;
    }
    ++n_ovf;
  }
  return n_ovf;
}

/* Inverse of the pack: dense g [T][F] from TwELL slots (non-overflow rows)
 * and the dense backup rows (overflow rows). */
void oracle_twell_unpack(int T, int F, int C, int K, const uint8_t *idx, const double *val,
                         const uint8_t *nnz, const uint8_t *row_ovf, const int32_t *ovf_rows,
                         int n_ovf, const double *g_fb, double *g) {
  int nt = F / C;
  memset(g, 0, sizeof(double) * (size_t)T * F);
  for (int t = 0; t < T; ++t) {
    if (row_ovf[t]) {
      for (int i = 0; i < n_ovf; ++i)
        if (ovf_rows[i] == t) memcpy(g + (size_t)t * F, g_fb + (size_t)i * F, sizeof(double) * F);
      continue;
    }
    for (int j = 0; j < nt; ++j) {
      int cnt = nnz[(size_t)j * T + t];
      size_t s0 = ((size_t)j * T + t) * (size_t)K;
      for (int k = 0; k < cnt && k < K; ++k)
        g[(size_t)t * F + (size_t)j * C + idx[s0 + k]] = val[s0 + k];
    }
  }
}

/* Dense FFN (the definition the sparse path must reproduce):
 *   g = round(ReLU(z)), u = x . Wu[n] (gated), h = g * u (gated) or g,
 *   y[t] = sum_{n ascending} h[t][n] * Wd[n].
 * Wu NULL selects the plain (non-gated) FFN.  y [T][D]; h_out [T][F] or NULL. */
void oracle_ffn_dense(int T, int D, int F, int dt, int q, const void *x, const void *Wg,
                      const float *bg, const float *rb, const void *Wu, const void *Wd,
                      double *y, double *h_out) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double *yt = y + (size_t)t * D;
    for (int d = 0; d < D; ++d) yt[d] = 0.0;
    for (int n = 0; n < F; ++n) {
      double zz = dot(x, dt, (size_t)t * D, Wg, dt, (size_t)n * D, D) + (double)bg[n];
      if (rb) zz += (double)rb[t];
      double g = is_active(zz, q) ? quant(zz, q) : 0.0;
      double h = g;
      if (Wu) h = g * dot(x, dt, (size_t)t * D, Wu, dt, (size_t)n * D, D);
      if (h_out) h_out[(size_t)t * F + n] = h;
      for (int d = 0; d < D; ++d) yt[d] += h * ld(Wd, dt, (size_t)n * D + d);
    }
  }
}

/* Sparse FFN consuming TwELL + dense backup rows (section 2.B inference):
 * non-overflow rows visit only their slots (tile ascending, slot ascending =
 * column ascending); overflow rows use their dense backup row. */
void oracle_ffn_twell(int T, int D, int F, int C, int K, int dt, const void *x, const void *Wu,
                      const void *Wd, const uint8_t *idx, const double *val, const uint8_t *nnz,
                      const uint8_t *row_ovf, const int32_t *ovf_rows, int n_ovf,
                      const double *g_fb, double *y) {
  int nt = F / C;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double *yt = y + (size_t)t * D;
    for (int d = 0; d < D; ++d) yt[d] = 0.0;
    const double *grow = NULL;
    if (row_ovf[t])
      for (int i = 0; i < n_ovf; ++i)
        if (ovf_rows[i] == t) grow = g_fb + (size_t)i * F;
    for (int j = 0; j < nt; ++j) {
      int cnt = nnz[(size_t)j * T + t];
      size_t s0 = ((size_t)j * T + t) * (size_t)K;
      int lim = grow ? C : (cnt < K ? cnt : K);
      for (int k = 0; k < lim; ++k) {
        int n;
        double g;
        if (grow) {
          n = j * C + k;
          g = grow[n];
          if (g == 0.0) continue;
        } else {
          n = j * C + idx[s0 + k];
          g = val[s0 + k];
        }
        double h = g;
        if (Wu) h = g * dot(x, dt, (size_t)t * D, Wu, dt, (size_t)n * D, D);
        for (int d = 0; d < D; ++d) yt[d] += h * ld(Wd, dt, (size_t)n * D + d);
      }
    }
  }
}

/* Classic row-ELL, the comparison format (section 2.A contrasts TwELL with
 * ELLPACK): for each row, the positive entries of a dense activation matrix
 * h [T][F] (entries >= 0, stored values) over the whole hidden axis, in
 * ascending column order, padded to E entries (index 0xFFFF, value +0); nnz
 * = the row's true count; entries past E are dropped. */
void oracle_rowell_pack(int T, int F, int E, const double *h, uint16_t *idx, double *val,
                        int32_t *nnz) {
  for (int t = 0; t < T; ++t) {
    int cnt = 0;
    for (int k = 0; k < E; ++k) {
      idx[(size_t)t * E + k] = 0xFFFF;
      val[(size_t)t * E + k] = 0.0;
    }
    for (int n = 0; n < F; ++n) {
      double v = h[(size_t)t * F + n];
      if (!(v > 0.0)) continue;
      if (cnt < E) {
        idx[(size_t)t * E + cnt] = (uint16_t)n;
        val[(size_t)t * E + cnt] = v;
      }
      ++cnt;
    }
    nnz[t] = cnt;
  }
}

/* Up + down projection from row-ELL gate values (section 2.B inference, with
 * the row-ELL format): y[t] = sum over the row's first min(nnz, E) entries,
 * ascending, of h * W_down[n], h = g * (x[t] . W_up[n]) (gated) or g. */
void oracle_ffn_rowell(int T, int D, int E, int dt, const void *x, const void *Wu,
                       const void *Wd, const uint16_t *idx, const double *val,
                       const int32_t *nnz, double *y) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double *yt = y + (size_t)t * D;
    for (int d = 0; d < D; ++d) yt[d] = 0.0;
    int m = nnz[t] < E ? nnz[t] : E;
    for (int k = 0; k < m; ++k) {
      int n = idx[(size_t)t * E + k];
      double hh = val[(size_t)t * E + k];
      if (Wu) hh *= dot(x, dt, (size_t)t * D, Wu, dt, (size_t)n * D, D);
      for (int d = 0; d < D; ++d) yt[d] += hh * ld(Wd, dt, (size_t)n * D + d);
    }
  }
}

/* Backward of the FFN with the L1 term (section 2.B training):
 *   L = sum_t dy[t] . y[t] + lambda * sum_{t,n} |h[t][n]|
 *   dh  = dy[t] . Wd[n] + lambda * sign(h)
 *   dz  = [z > 0] * dh * u   (gated)   or [z > 0] * dh   (plain)
 *   du  = dh * g             (gated)
 *   dx[t]  = sum_n dz Wg[n] + du Wu[n]
 *   dWg[n] = sum_t dz x[t],  dbg[n] = sum_t dz,  dWu[n] = sum_t du x[t],
 *   dWd[n] = sum_t h dy[t]
 * g and u are the values the training forward saves for the backward,
 * rounded to the storage type q (the backward consumes the saved activations,
 * section 2.A hybrid format / section 4 training memory); the rounding is
 * treated as identity for differentiation.  tok_sel / neu_sel (NULL = all)
 * select which dx rows
 * and which dW rows are produced; outputs are packed in selection order:
 * dx [n_tok][D], dWg/dWu/dWd [n_neu][D], dbg [n_neu].  dWu may be NULL for
 * the plain FFN.  Every selected output is computed from the definition. */
void oracle_ffn_backward(int T, int D, int F, int dt, int q, const void *x, const void *Wg,
                         const float *bg, const float *rb, const void *Wu, const void *Wd,
                         const void *dy, double lambda, const int32_t *tok_sel, int n_tok,
                         const int32_t *neu_sel, int n_neu, double *dx, double *dWg,
                         double *dbg, double *dWu, double *dWd) {
  if (!tok_sel) n_tok = T;
  if (!neu_sel) n_neu = F;
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n_tok; ++i) {
    int t = tok_sel ? tok_sel[i] : i;
    double *dxt = dx + (size_t)i * D;
    for (int d = 0; d < D; ++d) dxt[d] = 0.0;
    for (int n = 0; n < F; ++n) {
      double zz = dot(x, dt, (size_t)t * D, Wg, dt, (size_t)n * D, D) + (double)bg[n];
      if (rb) zz += (double)rb[t];
      if (!is_active(zz, q)) continue; /* dz = du = 0 exactly */
      double g = quant(zz, q);
      /* u as the forward saved it: rounded to the storage type, like g */
      double u = Wu ? quant(dot(x, dt, (size_t)t * D, Wu, dt, (size_t)n * D, D), q) : 1.0;
      double h = Wu ? g * u : g;
      double dh = dot(dy, dt, (size_t)t * D, Wd, dt, (size_t)n * D, D) + lambda * sgn(h);
      double dz = Wu ? dh * u : dh;
      double du = dh * g;
      for (int d = 0; d < D; ++d) {
        dxt[d] += dz * ld(Wg, dt, (size_t)n * D + d);
        if (Wu) dxt[d] += du * ld(Wu, dt, (size_t)n * D + d);
      }
    }
  }
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n_neu; ++i) {
    int n = neu_sel ? neu_sel[i] : i;
    double *gw = dWg + (size_t)i * D, *dw = dWd + (size_t)i * D;
    double *uw = dWu ? dWu + (size_t)i * D : NULL;
    double sb = 0.0;
    for (int d = 0; d < D; ++d) {
      gw[d] = 0.0;
      dw[d] = 0.0;
      if (uw) uw[d] = 0.0;
    }
    for (int t = 0; t < T; ++t) {
      double zz = dot(x, dt, (size_t)t * D, Wg, dt, (size_t)n * D, D) + (double)bg[n];
      if (rb) zz += (double)rb[t];
      if (!is_active(zz, q)) continue;
      double g = quant(zz, q);
      double u = Wu ? quant(dot(x, dt, (size_t)t * D, Wu, dt, (size_t)n * D, D), q) : 1.0;
      double h = Wu ? g * u : g;
      double dh = dot(dy, dt, (size_t)t * D, Wd, dt, (size_t)n * D, D) + lambda * sgn(h);
      double dz = Wu ? dh * u : dh;
      double du = dh * g;
      sb += dz;
      for (int d = 0; d < D; ++d) {
        double xv = ld(x, dt, (size_t)t * D + d);
        gw[d] += dz * xv;
        if (uw) uw[d] += du * xv;
        dw[d] += h * ld(dy, dt, (size_t)t * D + d);
      }
    }
    dbg[i] = sb;
  }
}

/* Loss of the FFN with the L1 term, for finite-difference pins:
 * L = sum_t dy[t] . y[t] + lambda * sum |h|, with y, h as in oracle_ffn_dense. */
double oracle_ffn_loss(int T, int D, int F, int dt, int q, const void *x, const void *Wg,
                       const float *bg, const float *rb, const void *Wu, const void *Wd,
                       const void *dy, double lambda) {
  double *y = (double *)malloc(sizeof(double) * (size_t)T * D);
  double *h = (double *)malloc(sizeof(double) * (size_t)T * F);
  if (!y || !h) {
    free(y);
    free(h);
    return NAN;
  }
  oracle_ffn_dense(T, D, F, dt, q, x, Wg, bg, rb, Wu, Wd, y, h);
  double L = 0.0;
  for (size_t i = 0; i < (size_t)T * D; ++i) L += ld(dy, dt, i) * y[i];
  for (size_t i = 0; i < (size_t)T * F; ++i) L += lambda * fabs(h[i]);
  free(y);
  free(h);
  return L;
}

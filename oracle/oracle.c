/*
 * oracle.c -- plain, slow CPU oracle for causal prefill attention with FP8 e4m3
 * and BF16 inputs.  TEST INFRASTRUCTURE ONLY: it is loaded by the tests, by the
 * smoke check and by the CPU-baseline leg of the benchmark, never by the
 * product path.  It shares no code, header, table or constant generator with
 * the CUDA library.
 *
 * Sources (web articles on Zyphra's ZYFA kernels), cited by title and section:
 *   [ART-EN]  "Breaking the FP8 Attention Bottleneck on AMD MI355X: How Zyphra
 *             ZYFA Unleashes Performance"
 *   [ART-MTP] "Zyphra ZYFA: FP8 FlashAttention for AMD MI355X, Up to 1.76x Faster"
 *
 * Every function works in fp64 and follows one definition written out in full:
 *
 *   oracle_ref_fp64      -- softmax(scale * Q K^T, causal) V on the DEQUANTIZED
 *                           inputs, the quantity whose RMS error [ART-MTP]
 *                           "How accurate is ZYFA's FP8 attention?" reports.
 *   oracle_emul_leanp    -- the Lean-P scheme of [ART-MTP] "How does ZYFA work?":
 *                           probability codes from one multiply-add and an
 *                           integer conversion ("Lean P: one multiply-add instead
 *                           of an exponential"), a power-of-two scale per 64-key
 *                           block and a row sum over the rounded probabilities
 *                           ("Per-block scaling and a rounded row sum").
 *   oracle_emul_exact_fp8 -- the exact-softmax FP8 ablation: exact exponential
 *                           relative to the running row max, each probability
 *                           rounded to e4m3, row sum over the unrounded values
 *                           (the "hardware exponential" column of [ART-MTP]
 *                           "How does ZYFA compare with other attention kernels?").
 *   oracle_emul_bf16     -- the exact-softmax BF16 path ([ART-MTP] "TL;DR").
 *   oracle_emul_leanp_a3 -- O-2 under the second reading of the block scale:
 *                           the code grid anchored at the running row maximum
 *                           instead of at integer log2 values.
 *   The *_ex forms take the options of a flash_attn_func-style call ([ART-MTP]
 *   "TL;DR" names that interface): causal or not, descales per (batch, kv
 *   head) or per tensor, and a per-row log-sum-exp of the path's own row sum.
 *
 * Readings where the articles are silent or ambiguous:
 *   - e4m3 is OCP E4M3 (bias 7, max 448, S.1111.111 = NaN, no infinities).
 *   - scale = softmax_scale argument (1/sqrt(Dqk) by default), per-tensor fp32
 *     descales, query head h reads kv head floor(h*Hkv/Hq).
 *   - Lean-P: in "code units" u = 8*lambda*s with lambda = log2(e)*scale*dq*dk and
 *     s the dot product of the decoded codes.  For each 64-key block beta (keys
 *     64*beta .. 64*beta+63, causally unmasked ones only) with largest u = b,
 *     e = ceil(b/8) and every key's code is clamp(floor(u - 8e + C), 0, 126)
 *     with C = 8*(7+T), T = 7, so the block maximum lands in the binade just
 *     below 2^T.  The block's weight factor is 2^(e - T).  The code grid is
 *     anchored at integer log2 values, so the result does not depend on the
 *     order in which key blocks are visited.
 *   - the exact FP8 ablation and the BF16 path use a running max updated once
 *     per 128-key tile in ascending key order.
 *   - descales are finite and positive (amax/448 of a tensor, or 1); every
 *     definition rejects other values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

/* Lean-P constants: headroom exponent T and the code C of 2^T (e4m3 code of
 * 2^x is 8*(x+7) for normal values). */
#define LEANP_T 7
#define LEANP_C (8 * (7 + LEANP_T))
#define LEANP_BLOCK 64
#define TILE_KEYS 128

/* ---------------------------------------------------------------------------
 * Number formats, written from their definitions.
 * ------------------------------------------------------------------------- */

/* OCP E4M3: value = (-1)^s * 2^(e-7) * (1 + m/8) for e >= 1,
 *                   (-1)^s * 2^(-6)  * (m/8)     for e == 0. */
double oracle_e4m3_decode(unsigned code) {
  unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  double mag;
  if (e == 15u && m == 7u) return NAN;
  if (e == 0u)
    mag = ldexp((double)m, -9);
  else
    mag = ldexp(8.0 + (double)m, (int)e - 10);
  return s ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_decode(unsigned bits) {
  uint32_t w = ((uint32_t)(bits & 0xFFFFu)) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* Round |x| to a binary format with `mbits` fraction bits and smallest normal
 * exponent `emin` (gradual underflow below), ties to even; `maxval` saturates. */
static double round_format(double x, int mbits, int emin, double maxval) {
  if (x == 0.0 || isnan(x)) return x;
  double ax = fabs(x);
  int e2;
  frexp(ax, &e2); /* ax = f * 2^e2, f in [0.5, 1): leading bit has weight 2^(e2-1) */
  int lead = e2 - 1;
  if (lead < emin) lead = emin;
  double quantum = ldexp(1.0, lead - mbits);
  double q = ax / quantum; /* exact: division by a power of two */
  double r = floor(q);
  double frac = q - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  r *= quantum;
  if (r > maxval) r = maxval;
  return x < 0 ? -r : r;
}

/* e4m3 round-to-nearest-even with saturation to +-448. */
double oracle_e4m3_round(double x) { return round_format(x, 3, -6, 448.0); }

/* bf16 round-to-nearest-even (finite inputs in range). */
double oracle_bf16_round(double x) { return round_format(x, 7, -126, INFINITY); }

/* ---------------------------------------------------------------------------
 * Shared helpers for the attention definitions (all fp64).
 * ------------------------------------------------------------------------- */

typedef struct {
  int B, Hq, Hkv, S, Dqk, Dv;
} shape_t;

/* Options common to the attention definitions: descales (one value, or one
 * per (batch, kv head) in [B, Hkv] order), the causal flag (keys j <= i, else
 * all S keys) and an optional per-row log-sum-exp output. */
typedef struct {
  const double *dq, *dk, *dv;
  int per_bkv;
  int causal;
} opts_t;

static double dsc(const double *a, const opts_t *o, const shape_t *sh, int b, int h) {
  if (!o->per_bkv) return a[0];
  int g = (int)(((int64_t)h * sh->Hkv) / sh->Hq);
  return a[(int64_t)b * sh->Hkv + g];
}

/* The descales must be finite and positive: a descale is amax/448 of a
 * tensor (1 for an all-zero one), and the library takes the same contract. */
static int descales_valid(const opts_t *o, const shape_t *sh) {
  const int64_t n = o->per_bkv ? (int64_t)sh->B * sh->Hkv : 1;
  for (int64_t t = 0; t < n; ++t) {
    const double a = o->dq[t], b = o->dk[t], c = o->dv[t];
    if (!(isfinite(a) && a > 0.0 && isfinite(b) && b > 0.0 && isfinite(c) && c > 0.0)) return 0;
  }
  return 1;
}

/* Number of keys row i attends to. */
static int keys_of(const opts_t *o, const shape_t *sh, int i) { return o->causal ? i + 1 : sh->S; }

static int check_shape(const shape_t *sh) {
  if (sh->B < 1 || sh->Hq < 1 || sh->Hkv < 1 || sh->S < 0 || sh->Dqk < 1 || sh->Dv < 1)
    return ORACLE_BAD_ARG;
  if (sh->Hq % sh->Hkv != 0) return ORACLE_BAD_ARG;
  return ORACLE_OK;
}

/* Row list: either `rows` holds n triples (b, h, i) or rows == NULL and all
 * B*S*Hq rows are produced in [B, S, Hq] order. */
static void row_at(const shape_t *sh, const int64_t *rows, int64_t r, int *b, int *h, int *i) {
  if (rows) {
    *b = (int)rows[3 * r];
    *h = (int)rows[3 * r + 1];
    *i = (int)rows[3 * r + 2];
  } else {
    *h = (int)(r % sh->Hq);
    *i = (int)((r / sh->Hq) % sh->S);
    *b = (int)(r / ((int64_t)sh->Hq * sh->S));
  }
}

static int rows_valid(const shape_t *sh, const int64_t *rows, int64_t n) {
  if (!rows) return ORACLE_OK;
  for (int64_t r = 0; r < n; ++r) {
    if (rows[3 * r] < 0 || rows[3 * r] >= sh->B) return ORACLE_BAD_ARG;
    if (rows[3 * r + 1] < 0 || rows[3 * r + 1] >= sh->Hq) return ORACLE_BAD_ARG;
    if (rows[3 * r + 2] < 0 || rows[3 * r + 2] >= sh->S) return ORACLE_BAD_ARG;
  }
  return ORACLE_OK;
}

/* Element offsets in the BSHD layout. */
static int64_t off_bshd(int b, int s, int h, int H, int S, int D) {
  return (((int64_t)b * S + s) * H + h) * D;
}

/* Decoded element of an input tensor: e4m3 codes (is_bf16 == 0) or bf16 bits. */
static double in_val(const void *base, int64_t idx, int is_bf16) {
  if (is_bf16) return oracle_bf16_decode(((const uint16_t *)base)[idx]);
  return oracle_e4m3_decode(((const uint8_t *)base)[idx]);
}

/* s_j = sum_d q_d * k_jd over the decoded (not descaled) values, and
 * a_j = sum_d |q_d * k_jd| (used for the rounding-ambiguity band). */
static void dot_row(const void *q, const void *k, const shape_t *sh, int is_bf16, int b,
                    int h, int i, int j, double *s, double *a) {
  int g = (int)(((int64_t)h * sh->Hkv) / sh->Hq);
  int64_t qo = off_bshd(b, i, h, sh->Hq, sh->S, sh->Dqk);
  int64_t ko = off_bshd(b, j, g, sh->Hkv, sh->S, sh->Dqk);
  double acc = 0.0, aacc = 0.0;
  for (int d = 0; d < sh->Dqk; ++d) {
    double p = in_val(q, qo + d, is_bf16) * in_val(k, ko + d, is_bf16);
    acc += p;
    aacc += fabs(p);
  }
  *s = acc;
  if (a) *a = aacc;
}

static double v_val(const void *v, const shape_t *sh, int is_bf16, int b, int h, int j, int d) {
  int g = (int)(((int64_t)h * sh->Hkv) / sh->Hq);
  return in_val(v, off_bshd(b, j, g, sh->Hkv, sh->S, sh->Dv) + d, is_bf16);
}

/* ---------------------------------------------------------------------------
 * O-1: fp64 attention on the dequantized inputs.
 *   z_ij = scale * <dq*q_i, dk*k_j>  (j <= i if causal, else all j < S),
 *   w = softmax_j(z_i.),  out_i = sum_j w_ij * dv * v_j,
 *   lse_i = ln sum_j exp(z_ij)  (natural log of the unnormalised row sum).
 * ------------------------------------------------------------------------- */
static int ref_fp64_impl(const void *q, const void *k, const void *v, int is_bf16, opts_t o,
                         shape_t sh, double scale, const int64_t *rows, int64_t nrows,
                         double *out, double *lse) {
  if (check_shape(&sh) || rows_valid(&sh, rows, nrows)) return ORACLE_BAD_ARG;
  if (!descales_valid(&o, &sh)) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    int b, h, i;
    row_at(&sh, rows, r, &b, &h, &i);
    const int n = keys_of(&o, &sh, i);
    const double dqk = dsc(o.dq, &o, &sh, b, h) * dsc(o.dk, &o, &sh, b, h);
    const double dv = dsc(o.dv, &o, &sh, b, h);
    double *z = (double *)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
      double s;
      dot_row(q, k, &sh, is_bf16, b, h, i, j, &s, NULL);
      z[j] = scale * (dqk * s);
      if (z[j] > m) m = z[j];
    }
    double L = 0.0;
    for (int j = 0; j < n; ++j) {
      z[j] = exp(z[j] - m);
      L += z[j];
    }
    for (int d = 0; d < sh.Dv; ++d) {
      double acc = 0.0;
      for (int j = 0; j < n; ++j) acc += z[j] * (dv * v_val(v, &sh, is_bf16, b, h, j, d));
      out[r * sh.Dv + d] = acc / L;
    }
    if (lse) lse[r] = m + log(L);
    free(z);
  }
  return ORACLE_OK;
}

int oracle_ref_fp64(const uint8_t *q, const uint8_t *k, const uint8_t *v, double dq, double dk,
                    double dv, int B, int Hq, int Hkv, int S, int Dqk, int Dv, double scale,
                    const int64_t *rows, int64_t nrows, double *out) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  opts_t o = {&dq, &dk, &dv, 0, 1};
  return ref_fp64_impl(q, k, v, 0, o, sh, scale, rows, nrows, out, NULL);
}

int oracle_ref_fp64_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                         int Hkv, int S, int Dqk, int Dv, double scale, const int64_t *rows,
                         int64_t nrows, double *out) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  const double one = 1.0;
  opts_t o = {&one, &one, &one, 0, 1};
  return ref_fp64_impl(q, k, v, 1, o, sh, scale, rows, nrows, out, NULL);
}

/* General form: is_bf16 selects bf16 inputs (descales then ignored, pass
 * NULL); dq/dk/dv hold one value or B*Hkv values (per_bkv); lse optional. */
int oracle_ref_fp64_ex(const void *q, const void *k, const void *v, int is_bf16,
                       const double *dq, const double *dk, const double *dv, int per_bkv,
                       int causal, int B, int Hq, int Hkv, int S, int Dqk, int Dv,
                       double scale, const int64_t *rows, int64_t nrows, double *out,
                       double *lse) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  const double one = 1.0;
  opts_t o = {is_bf16 ? &one : dq, is_bf16 ? &one : dk, is_bf16 ? &one : dv,
              is_bf16 ? 0 : per_bkv, causal};
  if (!o.dq || !o.dk || !o.dv) return ORACLE_BAD_ARG;
  return ref_fp64_impl(q, k, v, is_bf16, o, sh, scale, rows, nrows, out, lse);
}

/* ---------------------------------------------------------------------------
 * O-2: Lean-P emulation.
 *
 * [ART-MTP] "Lean P: one multiply-add instead of an exponential": an e4m3 bit
 * pattern read as an integer grows by 8 when the value doubles, so the code of
 * 2^x is about 8x plus a constant; each probability code is one multiply-add
 * followed by an integer conversion.
 * [ART-MTP] "Per-block scaling and a rounded row sum": each 64-key block is
 * scaled by a power of two before rounding, the scale is removed inside the
 * P.V product, and the row is divided by the sum of the ROUNDED probabilities.
 *
 * Per row i and block beta (unmasked keys: j <= i, or all j < S non-causal):
 *   u_j   = 8 * lambda * s_j                                  (code units)
 *   e     = ceil(max_{j in beta} u_j / 8)                     (block exponent)
 *   c_j   = clamp(floor(u_j - 8e + C), 0, 126)                (Lean-P code)
 *   w_j   = dec(c_j) * 2^(e - T)                              (descaled weight)
 *   out_i = dv * sum_j w_j v_j / sum_j w_j
 * Weights are formed relative to 2^(E) with E the largest block exponent of
 * the row, a common factor that cancels.
 *
 * amb[r] (if non-NULL) bounds the normalised weight mass that may change when
 * an fp32 evaluation of u lands on the other side of a rounding decision:
 * every floor whose argument lies within kappa * 8*lambda*sum_d|q_d k_jd| of an
 * integer, and every block exponent whose argument lies within that band of an
 * integer, contributes |w(alternative) - w| / sum_j w_j.
 * ------------------------------------------------------------------------- */

static int leanp_code(double x) {
  double f = floor(x);
  if (f < 0.0) return 0;
  if (f > 126.0) return 126;
  return (int)f;
}

/* exact_p = 1 gives the diagnostic variant E: the same blocks, exponents and
 * rounded row sum, but each weight is the exact value 2^(u_j/8 - e + T)
 * rounded to e4m3 (nearest even) instead of the Lean-P code, so that E - A
 * measures the block scale and the rounded sum and Lean-P - E the code. */
static int leanp_impl(const uint8_t *q, const uint8_t *k, const uint8_t *v, opts_t o, shape_t sh,
                      double scale, const int64_t *rows, int64_t nrows, double kappa, double *out,
                      double *amb, double *lse, int exact_p) {
  if (check_shape(&sh) || rows_valid(&sh, rows, nrows)) return ORACLE_BAD_ARG;
  if (!descales_valid(&o, &sh)) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    int b, h, i;
    row_at(&sh, rows, r, &b, &h, &i);
    /* log2(e) * scale * dq * dk */
    const double lam = scale * dsc(o.dq, &o, &sh, b, h) * dsc(o.dk, &o, &sh, b, h) / log(2.0);
    const double dv = dsc(o.dv, &o, &sh, b, h);
    int n = keys_of(&o, &sh, i);
    int nblk = (n + LEANP_BLOCK - 1) / LEANP_BLOCK;
    double *u = (double *)malloc(sizeof(double) * (size_t)n);
    double *du = (double *)malloc(sizeof(double) * (size_t)n);
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    int *eb = (int *)malloc(sizeof(int) * (size_t)nblk);
    for (int j = 0; j < n; ++j) {
      double s, a;
      dot_row(q, k, &sh, 0, b, h, i, j, &s, &a);
      u[j] = 8.0 * lam * s;
      /* band: fp32 accumulation of the dot product (kappa * sum|q k|) plus the
       * fp32 rounding of the scale constant itself (a few units of 2^-24) */
      du[j] = kappa * 8.0 * fabs(lam) * a + fabs(u[j]) * ldexp(1.0, -21);
    }
    int E = INT32_MIN;
    for (int bb = 0; bb < nblk; ++bb) {
      int j0 = bb * LEANP_BLOCK, j1 = j0 + LEANP_BLOCK < n ? j0 + LEANP_BLOCK : n;
      double bmax = -INFINITY;
      for (int j = j0; j < j1; ++j)
        if (u[j] > bmax) bmax = u[j];
      eb[bb] = (int)ceil(bmax / 8.0);
      if (eb[bb] > E) E = eb[bb];
    }
    double L = 0.0, dmass = 0.0;
    for (int bb = 0; bb < nblk; ++bb) {
      int j0 = bb * LEANP_BLOCK, j1 = j0 + LEANP_BLOCK < n ? j0 + LEANP_BLOCK : n;
      double f = ldexp(1.0, eb[bb] - E - LEANP_T);
      for (int j = j0; j < j1; ++j) {
        double x = u[j] - 8.0 * eb[bb] + LEANP_C;
        if (exact_p) {
          double y = exp2(u[j] / 8.0 - eb[bb] + LEANP_T);
          w[j] = oracle_e4m3_round(y) * f;
          L += w[j];
          if (amb) {
            /* the nearest e4m3 may flip when y moves by the relative error of
             * its fp32 argument (du/8 binades) and of a 2^-20-accurate 2^x */
            double d = log(2.0) * du[j] / 8.0 + ldexp(1.0, -20);
            double lo = oracle_e4m3_round(y * (1.0 - d)), hi = oracle_e4m3_round(y * (1.0 + d));
            dmass += (hi - lo) * f;
          }
          continue;
        }
        int c = leanp_code(x);
        w[j] = oracle_e4m3_decode((unsigned)c) * f;
        L += w[j];
        if (amb) {
          double nr = floor(x + 0.5);
          if (fabs(x - nr) < du[j]) { /* floor may land on nr-1 or nr */
            int c_lo = leanp_code(nr - 0.5), c_hi = leanp_code(nr + 0.5);
            dmass += fabs(oracle_e4m3_decode((unsigned)c_hi) - oracle_e4m3_decode((unsigned)c_lo)) * f;
          }
        }
      }
      if (amb) {
        /* block exponent: ceil(bmax/8) may move by one if bmax/8 is near an integer */
        double bmax = -INFINITY, dbm = 0.0;
        for (int j = j0; j < j1; ++j)
          if (u[j] > bmax) { bmax = u[j]; dbm = du[j]; }
        double t = bmax / 8.0, nt = floor(t + 0.5);
        if (fabs(t - nt) < dbm / 8.0) {
          int ea = (int)nt, eb2 = (int)nt + 1; /* ceil is nt or nt+1 */
          double fa = ldexp(1.0, ea - E - LEANP_T), fb = ldexp(1.0, eb2 - E - LEANP_T);
          for (int j = j0; j < j1; ++j) {
            double wa, wb;
            if (exact_p) {
              wa = oracle_e4m3_round(exp2(u[j] / 8.0 - ea + LEANP_T)) * fa;
              wb = oracle_e4m3_round(exp2(u[j] / 8.0 - eb2 + LEANP_T)) * fb;
            } else {
              wa = oracle_e4m3_decode((unsigned)leanp_code(u[j] - 8.0 * ea + LEANP_C)) * fa;
              wb = oracle_e4m3_decode((unsigned)leanp_code(u[j] - 8.0 * eb2 + LEANP_C)) * fb;
            }
            dmass += fabs(wa - wb);
          }
        }
      }
    }
    for (int d = 0; d < sh.Dv; ++d) {
      double acc = 0.0;
      for (int j = 0; j < n; ++j) acc += w[j] * v_val(v, &sh, 0, b, h, j, d);
      out[r * sh.Dv + d] = dv * acc / L;
    }
    if (amb) amb[r] = dmass / L;
    /* the rounded row sum in absolute units: sum_j w_j * 2^E ~ sum_j e^(z_j) */
    if (lse) lse[r] = log(L) + E * log(2.0);
    free(u);
    free(du);
    free(w);
    free(eb);
  }
  return ORACLE_OK;
}

int oracle_emul_leanp(const uint8_t *q, const uint8_t *k, const uint8_t *v, double dq, double dk,
                      double dv, int B, int Hq, int Hkv, int S, int Dqk, int Dv, double scale,
                      const int64_t *rows, int64_t nrows, double kappa, double *out,
                      double *amb) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  opts_t o = {&dq, &dk, &dv, 0, 1};
  return leanp_impl(q, k, v, o, sh, scale, rows, nrows, kappa, out, amb, NULL, 0);
}

int oracle_emul_leanp_ex(const uint8_t *q, const uint8_t *k, const uint8_t *v, const double *dq,
                         const double *dk, const double *dv, int per_bkv, int causal, int B,
                         int Hq, int Hkv, int S, int Dqk, int Dv, double scale,
                         const int64_t *rows, int64_t nrows, double kappa, double *out,
                         double *amb, double *lse) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  if (!dq || !dk || !dv) return ORACLE_BAD_ARG;
  opts_t o = {dq, dk, dv, per_bkv, causal};
  return leanp_impl(q, k, v, o, sh, scale, rows, nrows, kappa, out, amb, lse, 0);
}

/* Diagnostic variant E: see leanp_impl.  amb as for Lean-P (kappa: the
 * relative bound of the fp32 dot product, as in oracle_emul_leanp). */
int oracle_emul_variant_e(const uint8_t *q, const uint8_t *k, const uint8_t *v, const double *dq,
                          const double *dk, const double *dv, int per_bkv, int causal, int B,
                          int Hq, int Hkv, int S, int Dqk, int Dv, double scale,
                          const int64_t *rows, int64_t nrows, double kappa, double *out,
                          double *amb, double *lse) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  if (!dq || !dk || !dv) return ORACLE_BAD_ARG;
  opts_t o = {dq, dk, dv, per_bkv, causal};
  return leanp_impl(q, k, v, o, sh, scale, rows, nrows, kappa, out, amb, lse, 1);
}

/* ---------------------------------------------------------------------------
 * O-2, second reading: Lean-P codes anchored at the row's running maximum.
 *
 * The same two passages as O-2 ([ART-MTP] "Lean P: one multiply-add instead of
 * an exponential", "Per-block scaling and a rounded row sum") leave open what
 * the power of two of a block is relative to.  O-2 anchors the code grid at
 * integer log2 values; this reading anchors it at the running row maximum m,
 * so that the key holding the maximum gets exactly the code of 2^T.  With
 * lambda = log2(e)*scale*dq*dk, T = 7, C = 56 + 8T = 112 and eps = 2^-6, per
 * row, for each 128-key tile in ascending order (keys j <= i, or all j < S):
 *   m_new = max(m, max_j s_j);  if m_new > m:  O, l *= 2^(lambda*(m - m_new))
 *           (0 when m = -inf), m = m_new
 *   for each 64-key block beta of the tile that holds an unmasked key:
 *     k   = floor(lambda * (m - max_{j in beta} s_j))             (integer >= 0)
 *     c_j = clamp(floor(8*lambda*(s_j - m) + 8k + C + eps), 0, 126)
 *     O  += 2^(-T-k) * sum_j dec(c_j) * v_j;   l += 2^(-T-k) * sum_j dec(c_j)
 *   out = dv * O / l;   lse = ln l + lambda * m * ln 2.
 * amb: as for O-2, with every code's band widened by twice the band of the
 * running maximum (its fp32 value shifts every code of the row), and the
 * block's k taken both ways when lambda*(m - block max) is within the band of
 * an integer.
 * ------------------------------------------------------------------------- */
#define LEANP_A3_EPS (1.0 / 64.0)

static double a3_weight(double u, double um, int k) {
  return oracle_e4m3_decode((unsigned)leanp_code(u - um + 8.0 * k + LEANP_C + LEANP_A3_EPS)) *
         ldexp(1.0, -LEANP_T - k);
}

static int leanp_a3_impl(const uint8_t *q, const uint8_t *k, const uint8_t *v, opts_t o,
                         shape_t sh, double scale, const int64_t *rows, int64_t nrows,
                         double kappa, double *out, double *amb, double *lse) {
  if (check_shape(&sh) || rows_valid(&sh, rows, nrows)) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    int b, h, i;
    row_at(&sh, rows, r, &b, &h, &i);
    const double lam = scale * dsc(o.dq, &o, &sh, b, h) * dsc(o.dk, &o, &sh, b, h) / log(2.0);
    const double dv = dsc(o.dv, &o, &sh, b, h);
    const int n = keys_of(&o, &sh, i);
    double *u = (double *)malloc(sizeof(double) * (size_t)n); /* 8*lambda*s_j, code units */
    double *du = (double *)malloc(sizeof(double) * (size_t)n);
    double *O = (double *)calloc((size_t)sh.Dv, sizeof(double));
    for (int j = 0; j < n; ++j) {
      double s, a;
      dot_row(q, k, &sh, 0, b, h, i, j, &s, &a);
      u[j] = 8.0 * lam * s;
      du[j] = kappa * 8.0 * fabs(lam) * a + fabs(u[j]) * ldexp(1.0, -21);
    }
    double um = -INFINITY, dum = 0.0, l = 0.0, dmass = 0.0;
    for (int t0 = 0; t0 < n; t0 += TILE_KEYS) {
      const int t1 = t0 + TILE_KEYS < n ? t0 + TILE_KEYS : n;
      double ut = -INFINITY, dut = 0.0;
      for (int j = t0; j < t1; ++j)
        if (u[j] > ut) { ut = u[j]; dut = du[j]; }
      if (ut > um) {
        const double alpha = um == -INFINITY ? 0.0 : exp2((um - ut) / 8.0);
        for (int d = 0; d < sh.Dv; ++d) O[d] *= alpha;
        l *= alpha;
        dmass *= alpha;
        um = ut;
        dum = dut;
      }
      for (int j0 = t0; j0 < t1; j0 += LEANP_BLOCK) {
        const int j1 = j0 + LEANP_BLOCK < t1 ? j0 + LEANP_BLOCK : t1;
        double bmax = -INFINITY, dbm = 0.0;
        for (int j = j0; j < j1; ++j)
          if (u[j] > bmax) { bmax = u[j]; dbm = du[j]; }
        const double y = (um - bmax) / 8.0; /* lambda * (m - block max) */
        const int kb = (int)floor(y);
        for (int j = j0; j < j1; ++j) {
          const double w = a3_weight(u[j], um, kb);
          l += w;
          for (int d = 0; d < sh.Dv; ++d) O[d] += w * v_val(v, &sh, 0, b, h, j, d);
          if (amb) {
            const double x = u[j] - um + 8.0 * kb + LEANP_C + LEANP_A3_EPS;
            const double nr = floor(x + 0.5);
            if (fabs(x - nr) < du[j] + 2.0 * dum) {
              const double f = ldexp(1.0, -LEANP_T - kb);
              dmass += fabs(oracle_e4m3_decode((unsigned)leanp_code(nr + 0.5)) -
                            oracle_e4m3_decode((unsigned)leanp_code(nr - 0.5))) * f;
            }
          }
        }
        if (amb) {
          const double ny = floor(y + 0.5);
          if (ny >= 1.0 && fabs(y - ny) < (dbm + dum) / 8.0) /* k may be ny - 1 or ny */
            for (int j = j0; j < j1; ++j)
              dmass += fabs(a3_weight(u[j], um, (int)ny) - a3_weight(u[j], um, (int)ny - 1));
        }
      }
    }
    for (int d = 0; d < sh.Dv; ++d) out[r * sh.Dv + d] = dv * O[d] / l;
    if (amb) amb[r] = dmass / l;
    if (lse) lse[r] = log(l) + um / 8.0 * log(2.0);
    free(u);
    free(du);
    free(O);
  }
  return ORACLE_OK;
}

int oracle_emul_leanp_a3(const uint8_t *q, const uint8_t *k, const uint8_t *v, const double *dq,
                         const double *dk, const double *dv, int per_bkv, int causal, int B,
                         int Hq, int Hkv, int S, int Dqk, int Dv, double scale,
                         const int64_t *rows, int64_t nrows, double kappa, double *out,
                         double *amb, double *lse) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  if (!dq || !dk || !dv) return ORACLE_BAD_ARG;
  opts_t o = {dq, dk, dv, per_bkv, causal};
  if (!descales_valid(&o, &sh)) return ORACLE_BAD_ARG;
  return leanp_a3_impl(q, k, v, o, sh, scale, rows, nrows, kappa, out, amb, lse);
}

/* ---------------------------------------------------------------------------
 * O-3 / O-4: exact-softmax paths with a running max (128-key tiles, ascending).
 *
 * For each tile t (keys 128t .. 128t+127, j <= i):
 *   m_new = max(m, max_j z_j);  alpha = 2^(lambda2*(m - m_new)) (0 if m = -inf)
 *   O = alpha*O, l = alpha*l, m = m_new
 *   p_j = 2^(lambda2*(s_j - m));  P_j = round_fmt(p_j)
 *   O += sum_j P_j v_j;  l += sum_j p_j   (the UNROUNDED probabilities)
 * out_i = dv * O / l.   lambda2 = log2(e) * scale * dq * dk.
 * FP8 ablation: round_fmt = e4m3 RNE.  BF16 path: round_fmt = bf16 RNE.
 * amb[r] (FP8 only): mass that may move when p_j lies within its fp32
 * evaluation band of an e4m3 rounding midpoint.
 * ------------------------------------------------------------------------- */
static int exact_impl(const void *q, const void *k, const void *v, int is_bf16, opts_t o,
                      shape_t sh, double scale, const int64_t *rows, int64_t nrows, double kappa,
                      double *out, double *amb, double *lse) {
  if (check_shape(&sh) || rows_valid(&sh, rows, nrows)) return ORACLE_BAD_ARG;
  if (!descales_valid(&o, &sh)) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    int b, h, i;
    row_at(&sh, rows, r, &b, &h, &i);
    const double lam = scale * dsc(o.dq, &o, &sh, b, h) * dsc(o.dk, &o, &sh, b, h) / log(2.0);
    const double dv = dsc(o.dv, &o, &sh, b, h);
    int n = keys_of(&o, &sh, i);
    double *x = (double *)malloc(sizeof(double) * (size_t)n); /* lambda2 * s_j (log2 units) */
    double *dx = (double *)malloc(sizeof(double) * (size_t)n);
    double *O = (double *)calloc((size_t)sh.Dv, sizeof(double));
    for (int j = 0; j < n; ++j) {
      double s, a;
      dot_row(q, k, &sh, is_bf16, b, h, i, j, &s, &a);
      x[j] = lam * s;
      dx[j] = kappa * fabs(lam) * a + fabs(x[j]) * ldexp(1.0, -21);
    }
    double m = -INFINITY, dm = 0.0, l = 0.0, dmass = 0.0;
    for (int t0 = 0; t0 < n; t0 += TILE_KEYS) {
      int t1 = t0 + TILE_KEYS < n ? t0 + TILE_KEYS : n;
      double mt = -INFINITY, dmt = 0.0;
      for (int j = t0; j < t1; ++j)
        if (x[j] > mt) { mt = x[j]; dmt = dx[j]; }
      if (mt > m) {
        double alpha = (m == -INFINITY) ? 0.0 : exp2(m - mt);
        for (int d = 0; d < sh.Dv; ++d) O[d] *= alpha;
        l *= alpha;
        dmass *= alpha;
        m = mt;
        dm = dmt;
      }
      for (int j = t0; j < t1; ++j) {
        double p = exp2(x[j] - m);
        double P = is_bf16 ? oracle_bf16_round(p) : oracle_e4m3_round(p);
        l += p;
        for (int d = 0; d < sh.Dv; ++d) O[d] += P * v_val(v, &sh, is_bf16, b, h, j, d);
        if (amb && !is_bf16 && p > 0.0) {
          /* relative band of p: the fp32 evaluation of x_j - m (bands of x_j
           * and of the max) plus the exponential's own error (< 2^-20) */
          double rel = log(2.0) * (dx[j] + dm) + ldexp(1.0, -20);
          double lo = oracle_e4m3_round(p * (1.0 - rel)), hi = oracle_e4m3_round(p * (1.0 + rel));
          dmass += fabs(hi - lo);
        }
      }
    }
    for (int d = 0; d < sh.Dv; ++d) out[r * sh.Dv + d] = dv * O[d] / l;
    if (amb) amb[r] = is_bf16 ? 0.0 : dmass / l;
    if (lse) lse[r] = (m + log2(l)) * log(2.0); /* row sum of the unrounded p */
    free(x);
    free(dx);
    free(O);
  }
  return ORACLE_OK;
}

int oracle_emul_exact_fp8(const uint8_t *q, const uint8_t *k, const uint8_t *v, double dq,
                          double dk, double dv, int B, int Hq, int Hkv, int S, int Dqk, int Dv,
                          double scale, const int64_t *rows, int64_t nrows, double kappa,
                          double *out, double *amb) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  opts_t o = {&dq, &dk, &dv, 0, 1};
  return exact_impl(q, k, v, 0, o, sh, scale, rows, nrows, kappa, out, amb, NULL);
}

int oracle_emul_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                     int Hkv, int S, int Dqk, int Dv, double scale, const int64_t *rows,
                     int64_t nrows, double *out) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  const double one = 1.0;
  opts_t o = {&one, &one, &one, 0, 1};
  return exact_impl(q, k, v, 1, o, sh, scale, rows, nrows, 0.0, out, NULL, NULL);
}

/* General form of both exact paths (is_bf16: the BF16 path, descales ignored). */
int oracle_emul_exact_ex(const void *q, const void *k, const void *v, int is_bf16,
                         const double *dq, const double *dk, const double *dv, int per_bkv,
                         int causal, int B, int Hq, int Hkv, int S, int Dqk, int Dv,
                         double scale, const int64_t *rows, int64_t nrows, double kappa,
                         double *out, double *amb, double *lse) {
  shape_t sh = {B, Hq, Hkv, S, Dqk, Dv};
  const double one = 1.0;
  opts_t o = {is_bf16 ? &one : dq, is_bf16 ? &one : dk, is_bf16 ? &one : dv,
              is_bf16 ? 0 : per_bkv, causal};
  if (!o.dq || !o.dk || !o.dv) return ORACLE_BAD_ARG;
  return exact_impl(q, k, v, is_bf16, o, sh, scale, rows, nrows, is_bf16 ? 0.0 : kappa, out,
                    is_bf16 ? NULL : amb, lse);
}

/* Lean-P code of a single code-unit argument x (exposed for the closed-form
 * pins): clamp(floor(x), 0, 126). */
int oracle_leanp_code(double x) { return leanp_code(x); }

int oracle_leanp_C(void) { return LEANP_C; }
int oracle_leanp_T(void) { return LEANP_T; }

/* ---------------------------------------------------------------------------
 * Quantisation of Q or K to per-tensor e4m3, optionally after a Hadamard
 * rotation of every head vector ([ART-MTP] "How accurate is ZYFA's FP8
 * attention?": most FP8 error comes from quantising Q, K and V, and a Hadamard
 * rotation of Q and K roughly halves it; the product Q K^T is unchanged by a
 * common orthogonal rotation).
 *
 * Definition (every step in fp32, the precision in which the codes are
 * decided on the GPU):
 *   x: n_vec vectors of D elements (bf16 bits or fp32), D in {128, 192}.
 *   rotate = 0: y = x.
 *   rotate = 1: y = the unnormalised Walsh-Hadamard transform of x in blocks
 *     of hb elements (hb = 128 for D = 128; three blocks of 64 for D = 192).
 *     Butterfly stages h = 1, 2, 4, ..., hb/2; in each, every pair (i, i+h)
 *     with i mod 2h < h becomes (x_i + x_{i+h}, x_i - x_{i+h}).
 *   amax = max |y| over the whole tensor; sc = 448 / amax (1 if amax = 0).
 *   code = e4m3 round-to-nearest-even of the fp32 product y * sc, saturated
 *     to +-448, keeping the sign of zero.
 *   descale = (amax / 448) * norm with norm = 1/sqrt(hb) (1 unrotated;
 *     amax = 0 gives 1 * norm), so dec(code) * descale approximates the
 *     orthonormal rotation of x.
 * ------------------------------------------------------------------------- */

/* e4m3 code of an fp32 value: round to nearest even, saturate, keep the sign. */
static uint8_t e4m3_code_of(float v) {
  const double r = round_format((double)v, 3, -6, 448.0);
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs(r);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
  int lead = e2 - 1;
  unsigned E, M;
  if (lead < -6) { /* subnormal: a = M * 2^-9 */
    E = 0;
    M = (unsigned)(a / ldexp(1.0, -9));
  } else {
    E = (unsigned)(lead + 7);
    M = (unsigned)(a / ldexp(1.0, lead) * 8.0) - 8u;
  }
  return (uint8_t)(sign | (E << 3) | M);
}

static float in_f32(const void *x, int x_is_f32, int64_t idx) {
  if (x_is_f32) return ((const float *)x)[idx];
  uint32_t bits = (uint32_t)((const uint16_t *)x)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

static void rotate_vec(float *y, int D) {
  const int hb = D == 192 ? 64 : D;
  for (int base = 0; base < D; base += hb)
    for (int h = 1; h < hb; h *= 2)
      for (int i = 0; i < hb; ++i)
        if ((i % (2 * h)) < h) {
          const float a = y[base + i], b = y[base + i + h];
          y[base + i] = a + b;
          y[base + i + h] = a - b;
        }
}

int oracle_quantize_e4m3(const void *x, int x_is_f32, int64_t n_vec, int D, int rotate,
                         uint8_t *codes, float *descale) {
  if (!x || !codes || !descale || n_vec < 0 || (D != 128 && D != 192)) return ORACLE_BAD_ARG;
  float amax = 0.0f;
  float y[192];
  for (int64_t v = 0; v < n_vec; ++v) {
    for (int d = 0; d < D; ++d) y[d] = in_f32(x, x_is_f32, v * D + d);
    if (rotate) rotate_vec(y, D);
    for (int d = 0; d < D; ++d)
      if (fabsf(y[d]) > amax) amax = fabsf(y[d]);
  }
  const float sc = amax > 0.0f ? 448.0f / amax : 1.0f;
  for (int64_t v = 0; v < n_vec; ++v) {
    for (int d = 0; d < D; ++d) y[d] = in_f32(x, x_is_f32, v * D + d);
    if (rotate) rotate_vec(y, D);
    for (int d = 0; d < D; ++d) {
      const float t = y[d] * sc;
      codes[v * D + d] = e4m3_code_of(t);
    }
  }
  const float norm = !rotate ? 1.0f : (D == 192 ? 0.125f : 0.0883883476483184405501f);
  const float base = amax > 0.0f ? amax / 448.0f : 1.0f;
  *descale = base * norm;
  return ORACLE_OK;
}

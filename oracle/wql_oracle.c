/*
 * wql_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU restatement of the weight-only quantised lm_head path.
 * Only the tests, the smoke check and the bench's CPU-baseline leg may load
 * it; the product library never links, loads or calls anything here, and
 * this file includes nothing from the product sources.
 *
 * What it follows (page titles and sections):
 *  - radiance_lmhead_int4.py, module constants and quantize_int4_rows():
 *    symmetric per-group int4, q in [-8, 7], scale from amax times r/7,
 *    clamped below at 1e-8, rounded to the storage dtype BEFORE q is chosen,
 *    q = round-half-even(w / s) clamped, nibble = q + 8; with the "mse" clip
 *    the ratios 1.0, 0.95, 0.9, 0.85, 0.8 are tried in that order and a
 *    ratio replaces the kept one only when its squared error is strictly
 *    smaller.
 *  - "Fused WNA16 GEMM for tied quantized lm_head logits", Purpose: the
 *    weight is packed along the hidden (input) dimension, eight codes per
 *    32-bit word (radiance_lmhead_int4.py: [N, K/8] int32); the in-word order
 *    the pages use is not defined there, so this library defines its own
 *    (see Packing below); the logits are
 *    X . dequant(Wq)^T.  Perf-evals table rows "W8-g128" and the reviewer
 *    comment (item 1) for int8 weights with per-group or per-row scales.
 *  - same page, reviewer comment item 2: take the top-K of the quantised
 *    logits, recompute those K rows exactly from the unquantised weight and
 *    scatter them back.
 *
 * Arithmetic (where the pages leave a step open, the reading is stated):
 *  - scale:   s = RN_sdtype(max(fl32(amax) *f32 fl32(r/qmax), 1e-8f)),
 *             qmax = 7 (int4) or 127 (int8); RTN uses r = 1.0 only.
 *  - code:    q = clamp(rint_even(w_f32 /f32 s_f32), qmin, qmax); if the
 *             rounded scale is zero (fp16 underflow) the group's q are all 0.
 *  - MSE:     err_r = sum over the group, k ascending, of (q*s - w)^2 in
 *             binary64, added one term at a time.
 *  - logits:  sum_k x[m,k] * (q[n,k] * s[n,g(k)]) in binary64, k ascending,
 *             plus bias[n]; A[m,n] = sum_k |x[m,k] * w[n,k]| is returned for
 *             the tolerance 1e-3 + 2e-3 * A.
 *  - top-K:   value descending, index ascending on equal values.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread (no fast-math),
 * so every float operation is the IEEE operation written.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

/* ------------------------------------------------------------------------ */
/* binary16 / bfloat16 <-> binary64, written from the IEEE 754 definitions.  */
/* ------------------------------------------------------------------------ */

/* Round the finite double |v| to a binary format with `p` significant bits,
 * minimum normal exponent `emin` and maximum exponent `emax`, ties to even.
 * Returns +inf on overflow. */
static double round_to_format(double v, int p, int emin, int emax) {
  double a = fabs(v);
  if (a == 0.0) return 0.0;
  int e;
  frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) -> exponent e-1 */
  int ex = e - 1;
  if (ex < emin) ex = emin;             /* subnormal range: fixed quantum */
  double quantum = ldexp(1.0, ex - (p - 1));
  double units = a / quantum;           /* exact: power-of-two scaling */
  double r = nearbyint(units);          /* default mode: ties to even */
  double out = r * quantum;
  /* largest finite: (2 - 2^(1-p)) * 2^emax */
  double maxfin = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
  if (out > maxfin) return INFINITY;
  return out;
}

static uint16_t encode_format(double v_signed, int p, int emin, int emax,
                              int expbits) {
  int neg = signbit(v_signed) ? 1 : 0;
  double a = fabs(v_signed);
  uint32_t sign = (uint32_t)neg << 15;
  int mbits = p - 1;
  int bias = (1 << (expbits - 1)) - 1;
  if (isnan(v_signed)) return (uint16_t)(sign | (((1u << expbits) - 1) << mbits) | (1u << (mbits - 1)));
  if (isinf(a)) return (uint16_t)(sign | (((1u << expbits) - 1) << mbits));
  if (a == 0.0) return (uint16_t)sign;
  int e;
  frexp(a, &e);
  int ex = e - 1;
  if (ex < emin) { /* subnormal */
    double units = a / ldexp(1.0, emin - mbits);
    return (uint16_t)(sign | (uint32_t)units);
  }
  double frac = a / ldexp(1.0, ex) - 1.0;         /* in [0, 1) */
  uint32_t mant = (uint32_t)(frac * (double)(1u << mbits));
  (void)emax;
  return (uint16_t)(sign | ((uint32_t)(ex + bias) << mbits) | mant);
}

uint16_t oracle_f32_to_f16(float f) {
  double v = (double)f;
  if (isnan(v)) return encode_format(v, 11, -14, 15, 5);
  double r = round_to_format(v, 11, -14, 15);
  return encode_format(copysign(r, v), 11, -14, 15, 5);
}

uint16_t oracle_f32_to_bf16(float f) {
  double v = (double)f;
  if (isnan(v)) return encode_format(v, 8, -126, 127, 8);
  double r = round_to_format(v, 8, -126, 127);
  return encode_format(copysign(r, v), 8, -126, 127, 8);
}

static double decode_format(uint16_t bits, int mbits, int expbits) {
  int neg = (bits >> 15) & 1;
  uint32_t e = (bits >> mbits) & ((1u << expbits) - 1);
  uint32_t mant = bits & ((1u << mbits) - 1);
  int bias = (1 << (expbits - 1)) - 1;
  double v;
  if (e == 0) {
    v = ldexp((double)mant, 1 - bias - mbits);
  } else if (e == (1u << expbits) - 1) {
    v = mant ? NAN : INFINITY;
  } else {
    v = ldexp(1.0 + (double)mant / (double)(1u << mbits), (int)e - bias);
  }
  return neg ? -v : v;
}

double oracle_f16_to_f64(uint16_t b) { return decode_format(b, 10, 5); }
double oracle_bf16_to_f64(uint16_t b) { return decode_format(b, 7, 8); }

static double load_elem(const void* base, int dtype, int64_t i) {
  switch (dtype) {
    case OR_F32: return (double)((const float*)base)[i];
    case OR_F16: return oracle_f16_to_f64(((const uint16_t*)base)[i]);
    default:     return oracle_bf16_to_f64(((const uint16_t*)base)[i]);
  }
}

static uint16_t store_scale(float s, int scale_dtype) {
  return scale_dtype == OR_F16 ? oracle_f32_to_f16(s) : oracle_f32_to_bf16(s);
}

static double scale_value(uint16_t bits, int scale_dtype) {
  return scale_dtype == OR_F16 ? oracle_f16_to_f64(bits) : oracle_bf16_to_f64(bits);
}

/* ------------------------------------------------------------------------ */
/* Quantiser (radiance_lmhead_int4.py, quantize_int4_rows; int8 variant).    */
/* ------------------------------------------------------------------------ */

static const double kClipRatios[5] = {1.0, 0.95, 0.9, 0.85, 0.8};

/* w: n*k values (row-major) of w_dtype.  group == 0 means one scale per row.
 * q_out: n*k signed codes.  scales_out: n*(k/group) storage-dtype bits.
 * ratio_out (nullable): index of the chosen clip ratio per group.
 * Returns 0, or -1 on bad arguments. */
static int quantize_rows(const void* w, int w_dtype, int64_t row_begin, int64_t row_end,
                         int64_t k, int bits, int group, int scale_dtype, int clip,
                         int8_t* q_out, uint16_t* scales_out, int8_t* ratio_out) {
  if (bits != 4 && bits != 8) return -1;
  int64_t g = group == 0 ? k : group;
  if (g <= 0 || k % g != 0) return -1;
  const int qmax = bits == 4 ? 7 : 127;
  const int qmin = bits == 4 ? -8 : -127;
  const int nratios = clip ? 5 : 1;
  const int64_t ngroups = k / g;
  int8_t* qtry = (int8_t*)malloc((size_t)g);
  float* wbuf = (float*)malloc((size_t)g * sizeof(float));
  if (!qtry || !wbuf) { free(qtry); free(wbuf); return -1; }
  for (int64_t row = row_begin; row < row_end; ++row) {
    for (int64_t gi = 0; gi < ngroups; ++gi) {
      const int64_t base = row * k + gi * g;
      /* the group's values, widened exactly to fp32 */
      for (int64_t j = 0; j < g; ++j) wbuf[j] = (float)load_elem(w, w_dtype, base + j);
      /* amax over the group, in fp32 (exact: max of magnitudes) */
      float amax = 0.0f;
      for (int64_t j = 0; j < g; ++j) {
        float a = fabsf(wbuf[j]);
        if (a > amax) amax = a;
      }
      double best_err = 0.0;
      int best_r = -1;
      uint16_t best_sbits = 0;
      for (int ri = 0; ri < nratios; ++ri) {
        float c = (float)(kClipRatios[ri] / (double)qmax);
        float prod = amax * c;                      /* fp32, round to nearest */
        if (prod < 1e-8f) prod = 1e-8f;             /* zero-group guard */
        uint16_t sbits = store_scale(prod, scale_dtype);
        float s = (float)scale_value(sbits, scale_dtype); /* exact widening */
        double err = 0.0;
        for (int64_t j = 0; j < g; ++j) {
          float wv = wbuf[j];
          int q;
          if (s == 0.0f) {
            q = 0;
          } else {
            float t = wv / s;                       /* IEEE fp32 division */
            float rq = rintf(t);                    /* ties to even */
            if (rq > (float)qmax) rq = (float)qmax;
            if (rq < (float)qmin) rq = (float)qmin;
            q = (int)rq;
          }
          qtry[j] = (int8_t)q;
          if (nratios > 1) {
            double d = (double)q * (double)s - (double)wv;
            err = err + d * d;
          }
        }
        if (best_r < 0 || err < best_err) {
          best_err = err;
          best_r = ri;
          best_sbits = sbits;
          memcpy(q_out + base, qtry, (size_t)g);
        }
      }
      scales_out[row * ngroups + gi] = best_sbits;
      if (ratio_out) ratio_out[row * ngroups + gi] = (int8_t)best_r;
    }
  }
  free(qtry);
  free(wbuf);
  return 0;
}

typedef struct {
  const void* w; int w_dtype; int64_t r0, r1, k; int bits, group, scale_dtype, clip;
  int8_t* q_out; uint16_t* scales_out; int8_t* ratio_out; int rc;
} quant_job;

static void* quant_worker(void* arg) {
  quant_job* J = (quant_job*)arg;
  J->rc = quantize_rows(J->w, J->w_dtype, J->r0, J->r1, J->k, J->bits, J->group,
                        J->scale_dtype, J->clip, J->q_out, J->scales_out, J->ratio_out);
  return NULL;
}

/* Rows are independent; nthreads >= 1 splits them into contiguous blocks. */
int oracle_quantize(const void* w, int w_dtype, int64_t n, int64_t k, int bits,
                    int group, int scale_dtype, int clip, int8_t* q_out,
                    uint16_t* scales_out, int8_t* ratio_out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int joined[256];
  quant_job jobs[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    int64_t r0 = t * per < n ? t * per : n;
    int64_t r1 = (t + 1) * per < n ? (t + 1) * per : n;
    quant_job J = {w, w_dtype, r0, r1, k, bits, group, scale_dtype, clip,
                   q_out, scales_out, ratio_out, 0};
    jobs[t] = J;
    joined[t] = 0;
    if (nthreads == 1 || pthread_create(&th[t], NULL, quant_worker, &jobs[t]) != 0) {
      quant_worker(&jobs[t]);
      joined[t] = 1;
    }
  }
  int rc = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (!joined[t]) pthread_join(th[t], NULL);
    if (jobs[t].rc != 0) rc = jobs[t].rc;
  }
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Packing: word i of a row holds elements 8i .. 8i+7; element 8i + j sits   */
/* in nibble position p(j) = 4*(j % 2) + j / 2, i.e. bits [4p, 4p+4): the    */
/* even elements fill bits 0..15 and the odd elements bits 16..31, each in   */
/* ascending order.                                                          */
/* ------------------------------------------------------------------------ */

static int nibble_pos(int j) { return 4 * (j % 2) + j / 2; }

int oracle_pack_int4(const uint8_t* nib, int64_t n, int64_t k, uint32_t* packed) {
  if (k % 8 != 0) return -1;
  for (int64_t r = 0; r < n; ++r)
    for (int64_t i = 0; i < k / 8; ++i) {
      uint32_t word = 0;
      for (int j = 0; j < 8; ++j)
        word |= ((uint32_t)(nib[r * k + 8 * i + j] & 15u)) << (4 * nibble_pos(j));
      packed[r * (k / 8) + i] = word;
    }
  return 0;
}

/* Pack signed int4 codes q in [-8, 7] as nibbles q + 8 (same layout). */
int oracle_pack_codes_int4(const int8_t* q, int64_t n, int64_t k, uint32_t* packed) {
  if (k % 8 != 0) return -1;
  for (int64_t r = 0; r < n; ++r)
    for (int64_t i = 0; i < k / 8; ++i) {
      uint32_t word = 0;
      for (int j = 0; j < 8; ++j)
        word |= ((uint32_t)(q[r * k + 8 * i + j] + 8) & 15u) << (4 * nibble_pos(j));
      packed[r * (k / 8) + i] = word;
    }
  return 0;
}

int oracle_unpack_int4(const uint32_t* packed, int64_t n, int64_t k, uint8_t* nib) {
  if (k % 8 != 0) return -1;
  for (int64_t r = 0; r < n; ++r)
    for (int64_t kk = 0; kk < k; ++kk) {
      uint32_t word = packed[r * (k / 8) + kk / 8];
      nib[r * k + kk] = (uint8_t)((word >> (4 * nibble_pos((int)(kk % 8)))) & 15u);
    }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Logits in binary64 from the packed weight (explicit unpack + dequant).    */
/* ------------------------------------------------------------------------ */

typedef struct {
  const void* x; int x_dtype; int64_t m, k;
  const void* qweight; int bits;
  const uint16_t* scales; int scale_dtype; int64_t group;
  int64_t n; const void* bias; int bias_dtype;
  const int64_t* rows; int64_t nrows;
  double* out; double* abs_out;
  int64_t r_begin, r_end;
} logits_job;

/* w[row, kk] = q * s, from the packed codes (explicit nibble unpack) and the
 * row's scales already widened to binary64 in srow. */
static double dequant(const logits_job* J, const double* srow, int64_t row, int64_t kk) {
  int q;
  if (J->bits == 4) {
    const uint32_t* P = (const uint32_t*)J->qweight;
    uint32_t word = P[row * (J->k / 8) + kk / 8];
    int nibble = (int)((word >> (4 * nibble_pos((int)(kk % 8)))) & 15u);
    q = nibble - 8;
  } else {
    q = (int)((const int8_t*)J->qweight)[row * J->k + kk];
  }
  return (double)q * srow[kk / J->group];
}

static void* logits_worker(void* arg) {
  const logits_job* J = (const logits_job*)arg;
  const int64_t ngroups = J->k / J->group;
  double* xd = (double*)malloc((size_t)(J->m * J->k) * sizeof(double));
  double* srow = (double*)malloc((size_t)ngroups * sizeof(double));
  double* wrow = (double*)malloc((size_t)J->k * sizeof(double));
  if (!xd || !srow || !wrow) { free(xd); free(srow); free(wrow); return (void*)1; }
  for (int64_t i = 0; i < J->m * J->k; ++i) xd[i] = load_elem(J->x, J->x_dtype, i);
  for (int64_t ri = J->r_begin; ri < J->r_end; ++ri) {
    int64_t row = J->rows ? J->rows[ri] : ri;
    for (int64_t gi = 0; gi < ngroups; ++gi)
      srow[gi] = scale_value(J->scales[row * ngroups + gi], J->scale_dtype);
    for (int64_t kk = 0; kk < J->k; ++kk) wrow[kk] = dequant(J, srow, row, kk);
    for (int64_t mi = 0; mi < J->m; ++mi) {
      const double* xr = xd + mi * J->k;
      double acc = 0.0, absacc = 0.0;
      for (int64_t kk = 0; kk < J->k; ++kk) {
        double p = xr[kk] * wrow[kk];
        acc = acc + p;
        absacc = absacc + fabs(p);
      }
      if (J->bias) acc = acc + load_elem(J->bias, J->bias_dtype, row);
      J->out[mi * J->nrows + ri] = acc;
      if (J->abs_out) J->abs_out[mi * J->nrows + ri] = absacc;
    }
  }
  free(xd); free(srow); free(wrow);
  return NULL;
}

/* x: [m, k] of x_dtype.  qweight: bits 4 -> uint32 [n, k/8]; bits 8 -> int8
 * [n, k].  scales: [n, k/group] (group 0 = per row).  bias: nullable [n].
 * rows: nullable list of nrows vocab rows; when NULL, nrows must equal n.
 * out / abs_out: [m, nrows].  nthreads >= 1 splits the rows. */
int oracle_logits(const void* x, int x_dtype, int64_t m, int64_t k,
                  const void* qweight, int bits, const uint16_t* scales,
                  int scale_dtype, int group, int64_t n, const void* bias,
                  int bias_dtype, const int64_t* rows, int64_t nrows,
                  double* out, double* abs_out, int nthreads) {
  int64_t g = group == 0 ? k : group;
  if ((bits != 4 && bits != 8) || g <= 0 || k % g != 0) return -1;
  if (bits == 4 && k % 8 != 0) return -1;
  if (!rows && nrows != n) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  logits_job base = {x, x_dtype, m, k, qweight, bits, scales, scale_dtype, g,
                     n, bias, bias_dtype, rows, nrows, out, abs_out, 0, 0};
  pthread_t th[256];
  int joined[256];
  logits_job jobs[256];
  int64_t per = (nrows + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = base;
    jobs[t].r_begin = t * per < nrows ? t * per : nrows;
    jobs[t].r_end = (t + 1) * per < nrows ? (t + 1) * per : nrows;
    joined[t] = 0;
    if (nthreads == 1 || pthread_create(&th[t], NULL, logits_worker, &jobs[t]) != 0) {
      logits_worker(&jobs[t]);   /* run inline if no thread could be made */
      joined[t] = 1;
    }
  }
  for (int t = 0; t < nthreads; ++t)
    if (!joined[t]) pthread_join(th[t], NULL);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-K (value desc, index asc) and exact rescoring of chosen rows.         */
/* ------------------------------------------------------------------------ */

int oracle_topk(const double* vals, int64_t m, int64_t n, int K,
                int32_t* idx_out, double* val_out) {
  if (K < 1) return -1;
  for (int64_t mi = 0; mi < m; ++mi) {
    int have = 0;
    for (int64_t j = 0; j < n; ++j) {
      double v = vals[mi * n + j];
      if (isnan(v)) continue;
      /* position where (v, j) belongs: after every entry that ranks higher */
      int pos = have;
      while (pos > 0) {
        double pv = val_out[mi * K + pos - 1];
        if (pv > v || (pv == v && idx_out[mi * K + pos - 1] < j)) break;
        --pos;
      }
      if (pos >= K) continue;
      int last = have < K ? have : K - 1;
      for (int t = last; t > pos; --t) {
        val_out[mi * K + t] = val_out[mi * K + t - 1];
        idx_out[mi * K + t] = idx_out[mi * K + t - 1];
      }
      val_out[mi * K + pos] = v;
      idx_out[mi * K + pos] = (int32_t)j;
      if (have < K) ++have;
    }
    for (int t = have; t < K; ++t) { val_out[mi * K + t] = -INFINITY; idx_out[mi * K + t] = -1; }
  }
  return 0;
}

/* out[m, K] = sum_k x[m,k] * wref[idx[m,K], k] (+ bias[idx]) in binary64. */
int oracle_rescore(const void* x, int x_dtype, int64_t m, int64_t k,
                   const void* wref, int wref_dtype, int64_t n,
                   const int32_t* idx, int K, const void* bias, int bias_dtype,
                   double* out, double* abs_out) {
  for (int64_t mi = 0; mi < m; ++mi)
    for (int t = 0; t < K; ++t) {
      int64_t row = idx[mi * K + t];
      if (row < 0 || row >= n) return -1;
      double acc = 0.0, absacc = 0.0;
      for (int64_t kk = 0; kk < k; ++kk) {
        double p = load_elem(x, x_dtype, mi * k + kk) *
                   load_elem(wref, wref_dtype, row * k + kk);
        acc = acc + p;
        absacc = absacc + fabs(p);
      }
      if (bias) acc = acc + load_elem(bias, bias_dtype, row);
      out[mi * K + t] = acc;
      if (abs_out) abs_out[mi * K + t] = absacc;
    }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Tied-embedding gather ("Fused WNA16 GEMM for tied quantized lm_head       */
/* logits", Purpose: the tied head's quantised weight is also the input      */
/* embedding, so a token's embedding row is that row of dequant(Wq)).        */
/* out[i, kk] = RN_out(q[ids[i], kk] * s[ids[i], kk / group]); the product   */
/* is taken in binary64 (exact: an 8-bit code times an 11- or 8-bit scale)   */
/* and rounded once to fp16 / bf16, ties to even.  An id outside [0, n)     */
/* gives a row of +0.  out: t*k storage-dtype bits.                          */
/* ------------------------------------------------------------------------ */
int oracle_embed_gather(const int32_t* ids, int64_t t, const void* qweight, int bits,
                        const uint16_t* scales, int scale_dtype, int64_t group, int64_t n,
                        int64_t k, int out_dtype, uint16_t* out) {
  if ((bits != 4 && bits != 8) || group <= 0 || k % group != 0 || k % 8 != 0) return -1;
  if (out_dtype != OR_F16 && out_dtype != OR_BF16) return -1;
  const int64_t ng = k / group;
  for (int64_t i = 0; i < t; ++i) {
    const int64_t row = ids[i];
    for (int64_t kk = 0; kk < k; ++kk) {
      double v = 0.0;
      if (row >= 0 && row < n) {
        int q;
        if (bits == 4) {
          const uint32_t word = ((const uint32_t*)qweight)[row * (k / 8) + kk / 8];
          q = (int)((word >> (4 * nibble_pos((int)(kk % 8)))) & 15u) - 8;
        } else {
          q = (int)((const int8_t*)qweight)[row * k + kk];
        }
        v = (double)q * scale_value(scales[row * ng + kk / group], scale_dtype);
      }
      if (out_dtype == OR_F16) {
        double r = round_to_format(v, 11, -14, 15);
        out[i * k + kk] = encode_format(copysign(r, v), 11, -14, 15, 5);
      } else {
        double r = round_to_format(v, 8, -126, 127);
        out[i * k + kk] = encode_format(copysign(r, v), 8, -126, 127, 8);
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* fp8 e4m3 per-row head (the fp8 lm_head the radiance_lmhead_int4.py       */
/* module docstring compares against: per-channel fp8).                     */
/* e4m3 ("fn" variant): sign, 4 exponent bits with bias 7, 3 mantissa bits; */
/* no infinities, the all-ones pattern is NaN, largest finite 448,          */
/* subnormals m * 2^-9.  Readings (the page gives no formula): the row's    */
/* scale is s = RN_sdtype(max(fl32(amax) *f32 fl32(1/448), 1e-8f)), rounded */
/* before the codes are chosen, as for int4; q = RN_e4m3(clamp(w /f32 s,    */
/* -448, 448)), ties to even; a zero scale gives q = 0.                      */
/* ------------------------------------------------------------------------ */

double oracle_e4m3_to_f64(uint8_t b) {
  const int neg = (b >> 7) & 1;
  const int e = (b >> 3) & 15;
  const int m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return neg ? -v : v;
}

uint8_t oracle_f64_to_e4m3(double v) {
  if (isnan(v)) return 0x7F;
  const int neg = signbit(v) ? 1 : 0;
  double a = fabs(v);
  if (a > 448.0) a = 448.0;                         /* saturate */
  /* 4 significant bits, minimum normal exponent -6: round_to_format handles
     the subnormal quantum 2^-9; results stay <= 448 (448 is representable) */
  const double r = round_to_format(a, 4, -6, 8);
  uint8_t bits;
  if (r == 0.0) {
    bits = 0;
  } else {
    int e;
    frexp(r, &e);
    int ex = e - 1;
    if (ex < -6) {
      bits = (uint8_t)(r / ldexp(1.0, -9));         /* subnormal: m * 2^-9 */
    } else {
      const int mant = (int)((r / ldexp(1.0, ex) - 1.0) * 8.0);
      bits = (uint8_t)(((ex + 7) << 3) | mant);
    }
  }
  return (uint8_t)(bits | (neg << 7));
}

/* w: n*k values of w_dtype; q_out: n*k e4m3 bytes; scales_out: n storage-dtype bits. */
int oracle_quantize_fp8(const void* w, int w_dtype, int64_t n, int64_t k, int scale_dtype,
                        uint8_t* q_out, uint16_t* scales_out) {
  if (k <= 0 || (scale_dtype != OR_F16 && scale_dtype != OR_BF16)) return -1;
  const float inv = (float)(1.0 / 448.0);
  for (int64_t r = 0; r < n; ++r) {
    float amax = 0.0f;
    for (int64_t kk = 0; kk < k; ++kk) {
      const float a = fabsf((float)load_elem(w, w_dtype, r * k + kk));
      if (a > amax) amax = a;
    }
    float s = amax * inv;
    if (s < 1e-8f) s = 1e-8f;
    const uint16_t sb = store_scale(s, scale_dtype);
    scales_out[r] = sb;
    const float sf = (float)scale_value(sb, scale_dtype);
    for (int64_t kk = 0; kk < k; ++kk) {
      if (sf == 0.0f) { q_out[r * k + kk] = 0; continue; }
      float t = (float)load_elem(w, w_dtype, r * k + kk) / sf;
      if (t > 448.0f) t = 448.0f;
      if (t < -448.0f) t = -448.0f;
      q_out[r * k + kk] = oracle_f64_to_e4m3((double)t);
    }
  }
  return 0;
}

/* out[m, n] = sum_k x[m,k] * (e4m3(q[n,k]) * s[n]) in binary64, k ascending;
 * abs_out (nullable) the matching sum |x * w|. */
int oracle_logits_fp8(const void* x, int x_dtype, int64_t m, int64_t k, const uint8_t* q,
                      const uint16_t* scales, int scale_dtype, int64_t n, double* out,
                      double* abs_out) {
  for (int64_t r = 0; r < n; ++r) {
    const double s = scale_value(scales[r], scale_dtype);
    for (int64_t mi = 0; mi < m; ++mi) {
      double acc = 0.0, absacc = 0.0;
      for (int64_t kk = 0; kk < k; ++kk) {
        const double p = load_elem(x, x_dtype, mi * k + kk) *
                         (oracle_e4m3_to_f64(q[r * k + kk]) * s);
        acc = acc + p;
        absacc = absacc + fabs(p);
      }
      out[mi * n + r] = acc;
      if (abs_out) abs_out[mi * n + r] = absacc;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Zero-point (asymmetric) int4 ("[CORE] Quantized lm-head Framework": its  */
/* test model's lm_head is quantised with sym=False).  The page gives no    */
/* formula; the reading is plain asymmetric round-to-nearest per group:     */
/*   s = RN_sdtype(max((fl32(max) -f32 fl32(min)) *f32 fl32(1/15), 1e-8f))   */
/*   with min <= 0 <= max over the group (so 0 is representable),            */
/*   z = clamp(rint_even(-min /f32 s), 0, 15)  (an integer zero point),     */
/*   q = clamp(rint_even(w /f32 s) + z, 0, 15), w ~ (q - z) * s.            */
/* A zero scale gives q = z = 0.  q_out: n*k codes 0..15; scales_out and    */
/* zeros_out: n*(k/group).                                                   */
/* ------------------------------------------------------------------------ */
int oracle_quantize_asym_int4(const void* w, int w_dtype, int64_t n, int64_t k, int group,
                              int scale_dtype, uint8_t* q_out, uint16_t* scales_out,
                              uint8_t* zeros_out) {
  if (group <= 0 || k % group != 0 || (scale_dtype != OR_F16 && scale_dtype != OR_BF16))
    return -1;
  const int64_t ng = k / group;
  const float inv15 = (float)(1.0 / 15.0);
  for (int64_t r = 0; r < n; ++r)
    for (int64_t g = 0; g < ng; ++g) {
      float lo = 0.0f, hi = 0.0f;
      for (int64_t j = 0; j < group; ++j) {
        const float v = (float)load_elem(w, w_dtype, r * k + g * group + j);
        if (v < lo) lo = v;
        if (v > hi) hi = v;
      }
      float s = (hi - lo) * inv15;
      if (s < 1e-8f) s = 1e-8f;
      const uint16_t sb = store_scale(s, scale_dtype);
      scales_out[r * ng + g] = sb;
      const float sf = (float)scale_value(sb, scale_dtype);
      int z = 0;
      if (sf != 0.0f) {
        z = (int)rintf(-lo / sf);
        if (z < 0) z = 0;
        if (z > 15) z = 15;
      }
      zeros_out[r * ng + g] = (uint8_t)z;
      for (int64_t j = 0; j < group; ++j) {
        const int64_t i = r * k + g * group + j;
        int q = 0;
        if (sf != 0.0f) {
          q = (int)rintf((float)load_elem(w, w_dtype, i) / sf) + z;
          if (q < 0) q = 0;
          if (q > 15) q = 15;
        }
        q_out[i] = (uint8_t)q;
      }
    }
  return 0;
}

/* out[m, n] = sum_k x[m,k] * ((q[n,k] - z[n,g]) * s[n,g]) in binary64, k ascending. */
int oracle_logits_asym_int4(const void* x, int x_dtype, int64_t m, int64_t k, const uint8_t* q,
                            const uint16_t* scales, const uint8_t* zeros, int scale_dtype,
                            int group, int64_t n, double* out, double* abs_out) {
  if (group <= 0 || k % group != 0) return -1;
  const int64_t ng = k / group;
  for (int64_t r = 0; r < n; ++r)
    for (int64_t mi = 0; mi < m; ++mi) {
      double acc = 0.0, absacc = 0.0;
      for (int64_t kk = 0; kk < k; ++kk) {
        const int64_t gi = r * ng + kk / group;
        const double wv = (double)((int)q[r * k + kk] - (int)zeros[gi]) *
                          scale_value(scales[gi], scale_dtype);
        const double p = load_elem(x, x_dtype, mi * k + kk) * wv;
        acc = acc + p;
        absacc = absacc + fabs(p);
      }
      out[mi * n + r] = acc;
      if (abs_out) abs_out[mi * n + r] = absacc;
    }
  return 0;
}

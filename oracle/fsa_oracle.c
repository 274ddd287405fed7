/*
 * fsa_oracle.c -- plain, slow, obviously-correct CPU oracle for MX block-scaled
 * attention with a reformulated softmax.  TEST INFRASTRUCTURE ONLY: nothing in
 * the product path links, loads or calls this file.  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * Sources (cited by title and section throughout):
 *   [FSA-brief]  "Fused-Softmax for efficient quantized attention",
 *                The Singularity Report, abstract paragraph.
 *   [FSA-digest] "Moving softmax to matrix operations speeds up AI inference by
 *                over 2x", zot.news research digest: summary, "Read it as",
 *                "How it works" figure.
 *   [EFQ]        "EFQ-Softmax: Exp-Free Quantization for Softmax",
 *                paper-with-me paper page, abstract.
 *   [OCP-MX]     OCP Microscaling Formats (MX) v1.0 (external standard for the
 *                element bit layouts; the pages name the formats only).
 *
 * Everything floating point is fp64 unless a step is defined in fp32 (the
 * emulation of the fused algorithm, whose fp32 steps are part of its
 * definition).
 *
 * Parity pins: every exported function is pinned by tests under tests/ that do
 * not re-type its formula (exhaustive code tables, closed forms, brute force,
 * invariants).  Parity unpinned: the pages fix neither the exp approximation of
 * [FSA-digest] "Read it as" nor the constants of the [EFQ] affine rule; the
 * readings implemented here are this project's, documented beside each step.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* O1: scalar codecs ([OCP-MX] element formats named in [FSA-brief] abstract   */
/* (MXFP8/MXFP6/MXFP4) and [EFQ] abstract (E2M1)).                              */
/* fmt: 0 = E4M3 (bias 7, 3 mantissa bits, max 448, NaN = S.1111.111, no inf)  */
/*      1 = E2M3 (bias 1, 3 mantissa bits, max 7.5, 6-bit code, no NaN/inf)    */
/*      2 = E2M1 (bias 1, 1 mantissa bit,  max 6,   4-bit code, no NaN/inf)    */
/*      3 = E8M0 scale (2^(code-127); 0xFF = NaN)                              */
/*      4 = E3M2 (bias 3, 2 mantissa bits, max 28,  6-bit code, no NaN/inf):   */
/*          the other MXFP6 element type of [OCP-MX]                            */
/*      5 = NVFP4 as an operand format: E2M1 element codes (as fmt 2) in blocks */
/*          of 16 with one E4M3 scale each (O2b below); not an element codec    */
/* ------------------------------------------------------------------------- */
typedef struct { int ebits, mbits, bias; double maxv; int sign_shift; } fmt_info;

static fmt_info info_of(int fmt) {
  fmt_info f;
  switch (fmt) {
    case 0: f.ebits = 4; f.mbits = 3; f.bias = 7; f.maxv = 448.0; f.sign_shift = 7; break;
    case 1: f.ebits = 2; f.mbits = 3; f.bias = 1; f.maxv = 7.5;   f.sign_shift = 5; break;
    case 4: f.ebits = 3; f.mbits = 2; f.bias = 3; f.maxv = 28.0;  f.sign_shift = 5; break;
    default: f.ebits = 2; f.mbits = 1; f.bias = 1; f.maxv = 6.0;  f.sign_shift = 3; break;
  }
  return f;
}

/* exponent of the largest normal power of two of each element format */
int orc_emax(int fmt) { return fmt == 0 ? 8 : (fmt == 4 ? 4 : 2); }

double orc_decode(int fmt, uint32_t code) {
  if (fmt == 3) {
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
  }
  fmt_info f = info_of(fmt);
  int s = (code >> f.sign_shift) & 1;
  uint32_t mag = code & ((1u << f.sign_shift) - 1);
  int e = (int)(mag >> f.mbits);
  int m = (int)(mag & ((1u << f.mbits) - 1));
  double v;
  if (fmt == 0 && e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, 1 - f.bias - f.mbits);            /* subnormal */
  else v = ldexp(1.0 + ldexp((double)m, -f.mbits), e - f.bias);
  return s ? -v : v;
}

/* Round x to the element grid, nearest with ties to even, saturating to the
 * largest finite magnitude ("satfinite"); the sign of x is kept, also for
 * results that round to zero.  NaN maps to the E4M3 NaN code (the other two
 * formats have none and are never given NaN). */
uint32_t orc_encode(int fmt, double x) {
  fmt_info f = info_of(fmt);
  uint32_t sbit = signbit(x) ? (1u << f.sign_shift) : 0u;
  if (isnan(x)) return fmt == 0 ? (sbit | 0x7F) : sbit;
  double a = fabs(x);
  int emin = 1 - f.bias;                       /* exponent of the smallest normal */
  double v;
  if (a >= f.maxv) {
    v = f.maxv;
  } else if (a == 0.0) {
    v = 0.0;
  } else {
    int ex; frexp(a, &ex);                     /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;                            /* floor(log2 a) */
    if (e < emin) e = emin;                    /* subnormal range shares the quantum */
    double q = ldexp(1.0, e - f.mbits);        /* grid spacing in this binade */
    v = nearbyint(a / q) * q;                  /* a/q is exact; rint = ties-to-even */
    if (v > f.maxv) v = f.maxv;
  }
  if (v == 0.0) return sbit;
  int ex; frexp(v, &ex);
  int e = ex - 1;
  uint32_t code;
  if (e < emin) {                              /* subnormal: exponent field 0 */
    code = (uint32_t)llround(v / ldexp(1.0, emin - f.mbits));
  } else {
    uint32_t m = (uint32_t)llround((v / ldexp(1.0, e) - 1.0) * (double)(1 << f.mbits));
    code = ((uint32_t)(e + f.bias) << f.mbits) | m;
  }
  return sbit | code;
}

static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float fl; memcpy(&fl, &u, 4);
  return (double)fl;
}

/* ------------------------------------------------------------------------- */
/* O2: MX quantisation of 32-element blocks ([FSA-brief] abstract names       */
/* MXFP8/6/4 GEMM operands; block size 32 and E8M0 scales per [OCP-MX]).       */
/* Block scale E = clamp(floor(log2 amax) - emax, -127, 127); element codes =  */
/* encode(x * 2^-E), exact in fp64.  amax = 0 gives E = -127.  A block with a  */
/* non-finite element gets the NaN scale byte 0xFF and NaN/zero codes.          */
/* x is addressed as x[r*row_stride + i*elem_stride]; a row of len elements is */
/* padded with zeros to a whole number of blocks.                               */
/* codes: one byte per element (logical code, fp4/fp6 in the low bits),        */
/*        row r at codes[r*codes_stride]; scales: scales[r*scales_stride + b]. */
/* ------------------------------------------------------------------------- */
void orc_mx_quantize(const uint16_t* x, int64_t nrows, int64_t len, int64_t row_stride,
                     int64_t elem_stride, int fmt, uint8_t* codes, int64_t codes_stride,
                     uint8_t* scales, int64_t scales_stride, int nthreads) {
  const int64_t nblk = (len + 31) / 32;
  const int emax = orc_emax(fmt);
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
  for (int64_t r = 0; r < nrows; ++r) {
    for (int64_t b = 0; b < nblk; ++b) {
      double xv[32];
      double amax = 0.0;
      int nonfinite = 0;
      for (int i = 0; i < 32; ++i) {
        int64_t idx = b * 32 + i;
        xv[i] = idx < len ? bf16_to_double(x[r * row_stride + idx * elem_stride]) : 0.0;
        if (!isfinite(xv[i])) nonfinite = 1;
        else if (fabs(xv[i]) > amax) amax = fabs(xv[i]);
      }
      uint8_t* c = codes + r * codes_stride + b * 32;
      if (nonfinite) {
        scales[r * scales_stride + b] = 0xFF;
        for (int i = 0; i < 32; ++i) c[i] = (uint8_t)(fmt == 0 ? 0x7F : 0);
        continue;
      }
      int E;
      if (amax == 0.0) {
        E = -127;
      } else {
        int ex; frexp(amax, &ex);
        E = (ex - 1) - emax;
        if (E < -127) E = -127;
        if (E > 127) E = 127;
      }
      scales[r * scales_stride + b] = (uint8_t)(E + 127);
      for (int i = 0; i < 32; ++i) c[i] = (uint8_t)orc_encode(fmt, ldexp(xv[i], -E));
    }
  }
}

/* ------------------------------------------------------------------------- */
/* O2b: NVFP4 quantisation (an operand format adjacent to the pages' MX ones:  */
/* NVIDIA's FP4 with E2M1 elements, one E4M3 scale per 16 consecutive         */
/* elements; the per-tensor second-level fp32 scale is not used, i.e. 1).      */
/* Per block: scale s = encode_E4M3(amax / 6) (nearest, ties to even,          */
/* saturating at 448; amax / 6 is taken in fp64); codes = encode_E2M1(x / s)   */
/* (nearest, ties to even, saturating at 6).  A scale that rounds to zero      */
/* gives zero codes; a block with a non-finite element gets the E4M3 NaN       */
/* scale byte 0x7F and zero codes.  Layout as orc_mx_quantize with 16-element  */
/* blocks: scales[r*scales_stride + b] for elements [16b, 16b + 16).           */
/* ------------------------------------------------------------------------- */
void orc_nvfp4_quantize(const uint16_t* x, int64_t nrows, int64_t len, int64_t row_stride,
                        int64_t elem_stride, uint8_t* codes, int64_t codes_stride,
                        uint8_t* scales, int64_t scales_stride, int nthreads) {
  const int64_t nblk = (len + 15) / 16;
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
  for (int64_t r = 0; r < nrows; ++r) {
    for (int64_t b = 0; b < nblk; ++b) {
      double xv[16];
      double amax = 0.0;
      int nonfinite = 0;
      for (int i = 0; i < 16; ++i) {
        int64_t idx = b * 16 + i;
        xv[i] = idx < len ? bf16_to_double(x[r * row_stride + idx * elem_stride]) : 0.0;
        if (!isfinite(xv[i])) nonfinite = 1;
        else if (fabs(xv[i]) > amax) amax = fabs(xv[i]);
      }
      uint8_t* c = codes + r * codes_stride + b * 16;
      if (nonfinite) {
        scales[r * scales_stride + b] = 0x7F;
        for (int i = 0; i < 16; ++i) c[i] = 0;
        continue;
      }
      const uint32_t sc = orc_encode(0, amax / 6.0);
      scales[r * scales_stride + b] = (uint8_t)sc;
      const double sv = orc_decode(0, sc);
      for (int i = 0; i < 16; ++i) c[i] = (uint8_t)(sv == 0.0 ? 0u : orc_encode(2, xv[i] / sv));
    }
  }
}

/* ------------------------------------------------------------------------- */
/* Problem geometry shared by the attention oracles.                            */
/* Query row id = (b*H + h)*Sq + i.  kv head = h / (H/Hkv) (grouped queries).  */
/* Key j is visible to query i iff j < Sk and (!causal || j <= i + Sk - Sq).   */
/* ------------------------------------------------------------------------- */
typedef struct { int B, H, Hkv, Sq, Sk, D, causal; } orc_geom;

static void row_coords(const orc_geom* g, int64_t row, int* b, int* h, int* i, int* kvh) {
  *i = (int)(row % g->Sq);
  int64_t bh = row / g->Sq;
  *h = (int)(bh % g->H);
  *b = (int)(bh / g->H);
  *kvh = *h / (g->H / g->Hkv);
}

static int last_visible(const orc_geom* g, int i) {      /* last visible key index, -1 if none */
  int last = g->Sk - 1;
  if (g->causal) {
    int lim = i + g->Sk - g->Sq;
    if (lim < last) last = lim;
  }
  return last;
}

/* Rows are processed in groups that share one (batch, kv head), so that the    */
/* dequantised keys and values of that head are built once per group.           */
typedef struct { int64_t key; int64_t idx; } orc_sortkey;

static int cmp_sortkey(const void* a, const void* b) {
  const orc_sortkey* x = (const orc_sortkey*)a; const orc_sortkey* y = (const orc_sortkey*)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  return x->idx < y->idx ? -1 : (x->idx > y->idx);
}

/* order[] receives row positions sorted by (b, kv head); returns the number of
 * groups and fills gstart[g] (gstart has room for nrows + 1 entries). */
static int64_t group_rows(const orc_geom* g, const int64_t* rows, int64_t nrows, int64_t* order, int64_t* gstart) {
  orc_sortkey* k = (orc_sortkey*)malloc(sizeof(orc_sortkey) * (size_t)(nrows > 0 ? nrows : 1));
  for (int64_t n = 0; n < nrows; ++n) {
    int b, h, i, kvh;
    row_coords(g, rows[n], &b, &h, &i, &kvh);
    k[n].key = (int64_t)b * g->Hkv + kvh;
    k[n].idx = n;
  }
  qsort(k, (size_t)nrows, sizeof(orc_sortkey), cmp_sortkey);
  int64_t ng = 0;
  for (int64_t n = 0; n < nrows; ++n) {
    order[n] = k[n].idx;
    if (n == 0 || k[n].key != k[n - 1].key) gstart[ng++] = n;
  }
  gstart[ng] = nrows;
  free(k);
  return ng;
}

/* ------------------------------------------------------------------------- */
/* Keys and values of one (batch, kv head), decoded to fp64 once per group:    */
/*   kh[j*D + d], vh[d*nk + j] for keys j < nk.                                  */
/* ------------------------------------------------------------------------- */
typedef struct { double* kh; double* vh; int nk; } orc_kv;

static void kv_free(orc_kv* kv) { free(kv->kh); free(kv->vh); kv->kh = kv->vh = NULL; }

static int group_nk(const orc_geom* g, const int64_t* rows, const int64_t* order, int64_t a, int64_t e) {
  int nk = 0;
  for (int64_t t = a; t < e; ++t) {
    int b, h, i, kvh;
    row_coords(g, rows[order[t]], &b, &h, &i, &kvh);
    int l = last_visible(g, i) + 1;
    if (l > nk) nk = l;
  }
  return nk;
}

static void kv_from_bf16(const uint16_t* k, const uint16_t* v, const orc_geom* g, int b, int kvh, int nk,
                         orc_kv* kv, int nthreads) {
  const int D = g->D;
  kv->nk = nk;
  kv->kh = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1) * D);
  kv->vh = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1) * D);
  const int64_t base = ((int64_t)b * g->Hkv + kvh) * (int64_t)g->Sk * D;
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
  for (int j = 0; j < nk; ++j)
    for (int d = 0; d < D; ++d) {
      kv->kh[(int64_t)j * D + d] = bf16_to_double(k[base + (int64_t)j * D + d]);
      kv->vh[(int64_t)d * nk + j] = bf16_to_double(v[base + (int64_t)j * D + d]);
    }
}

/* ------------------------------------------------------------------------- */
/* Dequantised MX operands (logical layouts, one code byte per element):       */
/*   q codes [B,H,Sq,D]  scales [B,H,Sq,D/32]        (blocks along D)           */
/*   k codes [B,Hkv,Sk,D] scales [B,Hkv,Sk,D/32]     (blocks along D)           */
/*   v codes [B,Hkv,D,Skp] scales [B,Hkv,D,Skp/32]   (V transposed, blocks along */
/*                                                   keys; Skp = Sk rounded up  */
/*                                                   to a multiple of 32)       */
/* ------------------------------------------------------------------------- */
typedef struct {
  const uint8_t *qc, *qs, *kc, *ks, *vc, *vs;
  int fmt_qk, fmt_v;
} orc_mx_operands;

static double deq(int fmt, uint8_t code, uint8_t scale) {
  return orc_decode(fmt, code) * orc_decode(3, scale);
}
/* element d of a row of the Q/K operand format: MX (32-element E8M0 blocks) or
 * NVFP4 (16-element E4M3 blocks) */
static double deq_qk(int fmt, const uint8_t* codes, const uint8_t* scales, int D, int d) {
  if (fmt == 5) return orc_decode(2, codes[d]) * orc_decode(0, scales[d / 16]);
  return deq(fmt, codes[d], scales[d / 32]);
}

static void q_hat(const orc_mx_operands* op, const orc_geom* g, int b, int h, int i, double* qh) {
  const int D = g->D, nb = op->fmt_qk == 5 ? D / 16 : D / 32;
  const int64_t qrow = ((int64_t)b * g->H + h) * g->Sq + i;
  for (int d = 0; d < D; ++d) qh[d] = deq_qk(op->fmt_qk, op->qc + qrow * D, op->qs + qrow * nb, D, d);
}

static void kv_from_mx(const orc_mx_operands* op, const orc_geom* g, int b, int kvh, int nk, orc_kv* kv,
                       int nthreads) {
  const int D = g->D, nb = op->fmt_qk == 5 ? D / 16 : D / 32;
  const int64_t Skp = ((int64_t)g->Sk + 31) / 32 * 32;
  const int64_t kvi = (int64_t)b * g->Hkv + kvh;
  kv->nk = nk;
  kv->kh = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1) * D);
  kv->vh = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1) * D);
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
  for (int j = 0; j < nk; ++j) {
    const int64_t krow = kvi * g->Sk + j;
    for (int d = 0; d < D; ++d) {
      kv->kh[(int64_t)j * D + d] = deq_qk(op->fmt_qk, op->kc + krow * D, op->ks + krow * nb, D, d);
      const int64_t vrow = kvi * D + d;
      kv->vh[(int64_t)d * nk + j] = deq(op->fmt_v, op->vc[vrow * Skp + j], op->vs[vrow * (Skp / 32) + j / 32]);
    }
  }
}

/* ------------------------------------------------------------------------- */
/* O3: exact attention, the "standard attention" path of the [FSA-digest]      */
/* "How it works" figure: softmax(scale * q k^T) v in fp64 from the unquantised */
/* bf16 inputs.  q [B,H,Sq,D], k/v [B,Hkv,Sk,D] raw bf16 bits.                  */
/* Rows with no visible key give a zero output row.                             */
/* ------------------------------------------------------------------------- */
void orc_attn_exact(const uint16_t* q, const uint16_t* k, const uint16_t* v, const orc_geom* g,
                    double scale, const int64_t* rows, int64_t nrows, double* out, int nthreads) {
  const int D = g->D;
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  int64_t* gstart = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  int64_t ng = group_rows(g, rows, nrows, order, gstart);
  for (int64_t gi = 0; gi < ng; ++gi) {
    int b0, h0, i0, kvh0;
    row_coords(g, rows[order[gstart[gi]]], &b0, &h0, &i0, &kvh0);
    orc_kv kv;
    kv_from_bf16(k, v, g, b0, kvh0, group_nk(g, rows, order, gstart[gi], gstart[gi + 1]), &kv, nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t t = gstart[gi]; t < gstart[gi + 1]; ++t) {
      int64_t n = order[t];
      int b, h, i, kvh;
      row_coords(g, rows[n], &b, &h, &i, &kvh);
      const uint16_t* qr = q + (((int64_t)b * g->H + h) * g->Sq + i) * D;
      int nk = last_visible(g, i) + 1;
      double* o = out + n * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (nk <= 0) continue;
      double* s = (double*)malloc(sizeof(double) * (size_t)nk);
      double* qd = (double*)malloc(sizeof(double) * (size_t)D);
      for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(qr[d]);
      double m = -INFINITY;
      for (int j = 0; j < nk; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qd[d] * kv.kh[(int64_t)j * D + d];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
      }
      double l = 0.0;
      for (int j = 0; j < nk; ++j) { s[j] = exp(s[j] - m); l += s[j]; }
      for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        const double* vr = kv.vh + (int64_t)d * kv.nk;
        for (int j = 0; j < nk; ++j) acc += s[j] * vr[j];
        o[d] = acc / l;
      }
      free(s); free(qd);
    }
    kv_free(&kv);
  }
  free(order); free(gstart);
}

/* ------------------------------------------------------------------------- */
/* O4: the error floor of [FSA-brief] abstract ("error floor set by          */
/* quantizing the GEMM operands") and the exp-then-quantize path of [EFQ]      */
/* abstract.  Scores from dequantised q_hat, k_hat in fp64, exact softmax       */
/* numerator p = exp(s - max) over visible keys; if quantize_p, p is MX-        */
/* quantised in 32-key blocks (aligned to key index multiples of 32) into       */
/* element format fmt_p by the O2 rule; O = sum p~ v_hat / sum p~.              */
/* ------------------------------------------------------------------------- */
void orc_attn_floor(const orc_mx_operands* op, const orc_geom* g, double scale, int fmt_p, int quantize_p,
                    const int64_t* rows, int64_t nrows, double* out, int nthreads) {
  const int D = g->D;
  const int emax = orc_emax(fmt_p);
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  int64_t* gstart = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  int64_t ng = group_rows(g, rows, nrows, order, gstart);
  for (int64_t gi = 0; gi < ng; ++gi) {
    int b0, h0, i0, kvh0;
    row_coords(g, rows[order[gstart[gi]]], &b0, &h0, &i0, &kvh0);
    orc_kv kv;
    kv_from_mx(op, g, b0, kvh0, group_nk(g, rows, order, gstart[gi], gstart[gi + 1]), &kv, nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t t = gstart[gi]; t < gstart[gi + 1]; ++t) {
      int64_t n = order[t];
      int b, h, i, kvh;
      row_coords(g, rows[n], &b, &h, &i, &kvh);
      int nk = last_visible(g, i) + 1;
      double* o = out + n * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (nk <= 0) continue;
      double* qh = (double*)malloc(sizeof(double) * D);
      double* p = (double*)malloc(sizeof(double) * (size_t)nk);
      q_hat(op, g, b, h, i, qh);
      double m = -INFINITY;
      for (int j = 0; j < nk; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qh[d] * kv.kh[(int64_t)j * D + d];
        p[j] = scale * acc;
        if (p[j] > m) m = p[j];
      }
      for (int j = 0; j < nk; ++j) p[j] = exp(p[j] - m);
      if (quantize_p) {
        for (int jb = 0; jb < nk; jb += 32) {
          int je = jb + 32 < nk ? jb + 32 : nk;
          double amax = 0.0;
          for (int j = jb; j < je; ++j) if (p[j] > amax) amax = p[j];
          int E = -127;
          if (amax > 0.0) {
            int ex; frexp(amax, &ex);
            E = (ex - 1) - emax;
            if (E < -127) E = -127;
            if (E > 127) E = 127;
          }
          for (int j = jb; j < je; ++j)
            p[j] = orc_decode(fmt_p, orc_encode(fmt_p, ldexp(p[j], -E))) * ldexp(1.0, E);
        }
      }
      double l = 0.0;
      for (int j = 0; j < nk; ++j) l += p[j];
      for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        const double* vr = kv.vh + (int64_t)d * kv.nk;
        for (int j = 0; j < nk; ++j) acc += p[j] * vr[j];
        o[d] = l > 0.0 ? acc / l : 0.0;
      }
      free(qh); free(p);
    }
    kv_free(&kv);
  }
  free(order); free(gstart);
}

/* ------------------------------------------------------------------------- */
/* exp2 approximation.  [FSA-digest] "Read it as": softmax "approximates the    */
/* exponential with a fast method"; the method is not given.  Reading: a Cody-  */
/* Waite split r = n + f, n = floor(r), f in [0,1); 2^f by the cubic that       */
/* interpolates 2^f at f = 0, 1/3, 2/3, 1 (coefficients solved in fp64 from     */
/* those four nodes, then rounded once to fp32), evaluated by Horner's rule     */
/* with fused multiply-adds; the result is scaled by 2^n exactly.  r is first   */
/* clamped below at -64 (any value under 2^-64 quantises to code 0 in every     */
/* element format).                                                             */
/* ------------------------------------------------------------------------- */
void orc_exp2_poly_coeffs(float c[4]) {
  double x[4] = {0.0, 1.0 / 3.0, 2.0 / 3.0, 1.0};
  double a[4][5];
  for (int r = 0; r < 4; ++r) {
    double p = 1.0;
    for (int k = 0; k < 4; ++k) { a[r][k] = p; p *= x[r]; }
    a[r][4] = exp2(x[r]);
  }
  for (int col = 0; col < 4; ++col) {            /* Gauss-Jordan with partial pivoting */
    int piv = col;
    for (int r = col + 1; r < 4; ++r) if (fabs(a[r][col]) > fabs(a[piv][col])) piv = r;
    for (int k = 0; k < 5; ++k) { double t = a[col][k]; a[col][k] = a[piv][k]; a[piv][k] = t; }
    for (int r = 0; r < 4; ++r) {
      if (r == col) continue;
      double fct = a[r][col] / a[col][col];
      for (int k = col; k < 5; ++k) a[r][k] -= fct * a[col][k];
    }
  }
  for (int k = 0; k < 4; ++k) c[k] = (float)(a[k][4] / a[k][k]);
}

float orc_exp2_poly(float r) {
  float c[4];
  orc_exp2_poly_coeffs(c);
  float rc = r < -64.0f ? -64.0f : r;                 /* also maps -inf to -64 */
  float n = floorf(rc);
  float f = rc - n;                                   /* exact */
  float p = fmaf(fmaf(fmaf(c[3], f, c[2]), f, c[1]), f, c[0]);
  return ldexpf(p, (int)n);
}

/* ------------------------------------------------------------------------- */
/* O5: step-by-step emulation of the fused MX attention forward:               */
/*  - [FSA-brief] abstract: QK^T and PV as MX GEMMs; softmax reformulated so   */
/*    its work folds into them.                                                  */
/*  - [FSA-digest] "Read it as" / "How it works": the maximum is frozen         */
/*    speculatively ("Speculative Max: Freeze max"), with a fallback when the   */
/*    guess is wrong; the exponential is approximated; "Exp + MX Quant" is       */
/*    fused; probabilities are summed on the matrix unit.                        */
/*  - [FSA-digest] summary: max subtraction and exponentiation folded into the  */
/*    score matrix multiply's output (one fused multiply-add per score).         */
/*  - [EFQ] abstract: per microscaling block an exponent-only scale from the    */
/*    local max, shifted scores mapped to a normalised residual domain, codes   */
/*    from one affine rule; the same operand feeds the P~V numerator and the    */
/*    P~1 denominator; final normalisation in high precision.                   */
/*                                                                              */
/* Per query row, over key tiles of 128 in ascending order (tiles with no       */
/* visible key for the row are skipped; they contribute nothing):               */
/*  1. s_j = fp32(exact dot(q_hat, k_hat_j))            (raw score, fp32)        */
/*  2. mx = max visible s_j;  x = fp32(mx * c), c = fp32(scale * log2 e)         */
/*  3. first tile: M = x (frozen max, log2 units)                                */
/*     later tile: if x > fp32(M + delta): fallback: M' = x, alpha = 2^(M - M'), */
/*                 O_acc *= alpha, l *= alpha, M = M', count++                   */
/*     (delta >= 0 is a margin on the fallback test only; M itself stays a      */
/*     rounded score product, so the block holding it has tmax = 0 exactly)     */
/*  4. per 32-key block: smax = max visible s; tmax = fp32(fp32(smax*c) - M);   */
/*     E = clamp(floor(tmax) - emax, -127, 127); bE = fp32(M + E);               */
/*     r_j = fmaf(s_j, c, -bE)  (residual: shifted log2 score minus E)           */
/*     exp path:  code = encode_fmt(exp2approx(r_j))                             */
/*     EFQ path:  the shift and the affine rule y = a r_j + b are one fused      */
/*                multiply-add on the raw score (the fold of [FSA-digest]        */
/*                summary): y = fmaf(s_j, A, Bk), A = fp32(a c), Bk =            */
/*                fp32(b - fp32(a bE)); code = clamp(round_half_even(y), 0, 7)    */
/*                (E2M1); the block exponent takes the reference point phi:      */
/*                E = clamp(floor(fp32(tmax + phi)) - emax, -127, 127).           */
/*     scale byte = E + 127; a block with no visible key: codes 0, scale 0x00    */
/*  5. O_acc += sum p~_j v_hat_j, l += sum p~_j with p~_j = dec(code) 2^E (fp64) */
/*  6. O = O_acc / l (0 if l == 0)                                               */
/* The per-element exp2approx is chosen by bit (j % 32) of mufu_mask: set ->     */
/* modelled as exact 2^r rounded to fp32 (the hardware approximation on the      */
/* GPU differs in the last bits); clear -> orc_exp2_poly (bit-reproducible).     */
/* fmt_p: 0 E4M3, 1 E2M3, 2 E2M1, 3 E2M1 by the EFQ rule, 4 E3M2.               */
/* ------------------------------------------------------------------------- */
typedef struct {
  float delta;        /* fallback margin, log2 units: fall back when x > M + delta */
  uint32_t mufu_mask; /* per position in a 32-block: 1 = hardware exp2 model */
  float beta;         /* EFQ affine offset b (default 2) */
  float efq_a;        /* EFQ affine slope a (default 2) */
  float phi;          /* reference point of the P block scale: E = floor(tmax + phi) - emax (default 0) */
  double s_perturb;   /* test knob: raw scores are fp32(dot * (1 + s_perturb)); 0 normally */
} orc_fsa_opts;

typedef struct {      /* optional per-row dumps, NULL to skip */
  float* s;           /* [nrows][Skp] raw scores (visible keys; masked -inf) */
  uint8_t* p_codes;   /* [nrows][Skp] P codes */
  uint8_t* p_scales;  /* [nrows][Skp/32] P scale bytes */
  float* m_frozen;    /* [nrows][ntiles] M after the tile's max step (NaN if skipped) */
  double* amb;        /* [nrows][D] bound on |O_kernel - O| from undetermined decisions (below) */
  const float* s_in;  /* optional input [nrows][Skp]: raw scores to use instead of step 1's
                         (a kernel's own scores, so that steps 2-6 can be checked given them) */
  uint8_t* p_alt;     /* [nrows][Skp] the code at the other end of the exp2 uncertainty
                         (AMB_X) for hardware-exp2 positions; equal to p_codes elsewhere */
  const uint8_t* p_in;/* optional input [nrows][Skp]: P codes to accumulate instead of step
                         5's (a kernel's own codes, once checked against p_codes / p_alt);
                         p_codes still reports the emulation's own */
} orc_fsa_dump;

/* Decisions the kernel takes in fp32 that this emulation cannot reproduce bit for
 * bit: the tensor core's fp32 score (its internal accumulation order is not
 * specified; modelled here as within AMB_S = 2^-21 of the sum of the absolute
 * 32-element block dot products, i.e. a few ulps of the largest partial sum), and
 * the hardware exp2 (within AMB_X = 2^-21 relative of 2^r).  A P code is
 * undetermined when the interval of inputs those uncertainties allow maps to more
 * than one code; a block exponent when its floor can go either way; a row when its
 * fallback test can.  For each undetermined code (or whole block) the possible
 * change dp of its value is added into B = sum dp and A_d = sum dp |v_jd|; a
 * fallback's factor 2^(M - M') carries the relative error of M, M' and the exp2
 * into everything accumulated before it; with
 * o the emulated output, |O_kernel_d - o_d| <= (A_d + B |o_d|) / (l - B), which is
 * written to amb (infinite for a row with an undetermined fallback). */
#define AMB_S 4.76837158203125e-07   /* 2^-21 */
#define AMB_X 4.76837158203125e-07   /* 2^-21 */

static float exp2_model(float r, int use_hw, const float* pc) {
  if (use_hw) return (float)exp2((double)r);
  float rc = r < -64.0f ? -64.0f : r;
  float n = floorf(rc);
  float f = rc - n;
  float p = fmaf(fmaf(fmaf(pc[3], f, pc[2]), f, pc[1]), f, pc[0]);
  return ldexpf(p, (int)n);
}

void orc_fsa_emulate(const orc_mx_operands* op, const orc_geom* g, float scale, int fmt_p,
                     const orc_fsa_opts* opt, const int64_t* rows, int64_t nrows, double* out,
                     int32_t* fallbacks, int32_t* tiles_visited, const orc_fsa_dump* dump, int nthreads) {
  const int D = g->D, BN = 128;
  const int64_t Skp = ((int64_t)g->Sk + 31) / 32 * 32;
  const int ntiles = (g->Sk + BN - 1) / BN;
  const float c = (float)((double)scale * 1.4426950408889634073599246810018921);  /* log2(e) */
  const int efq = fmt_p == 3;
  const int efmt = efq ? 2 : fmt_p;
  const int emax = orc_emax(efmt);
  const float a_c = opt->efq_a * c;               /* EFQ: fp32(a c) */
  const float phi = efq ? opt->phi : 0.0f;        /* the exp path keeps the OCP scale rule */
  float pc[4];
  orc_exp2_poly_coeffs(pc);
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  int64_t* gstart = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  int64_t ng = group_rows(g, rows, nrows, order, gstart);
  for (int64_t gi = 0; gi < ng; ++gi) {
    int b0, h0, i0, kvh0;
    row_coords(g, rows[order[gstart[gi]]], &b0, &h0, &i0, &kvh0);
    orc_kv kv;
    kv_from_mx(op, g, b0, kvh0, group_nk(g, rows, order, gstart[gi], gstart[gi + 1]), &kv, nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t t0 = gstart[gi]; t0 < gstart[gi + 1]; ++t0) {
      int64_t n = order[t0];
      int b, h, i, kvh;
      row_coords(g, rows[n], &b, &h, &i, &kvh);
      int nk = last_visible(g, i) + 1;
      double* o = out + n * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      int fb = 0, tv = 0;
      if (dump && dump->m_frozen) for (int t = 0; t < ntiles; ++t) dump->m_frozen[n * ntiles + t] = NAN;
      if (dump && dump->s) for (int64_t j = 0; j < Skp; ++j) dump->s[n * Skp + j] = -INFINITY;
      if (dump && dump->p_codes) memset(dump->p_codes + n * Skp, 0, (size_t)Skp);
      if (dump && dump->p_alt) memset(dump->p_alt + n * Skp, 0, (size_t)Skp);
      if (dump && dump->p_scales) memset(dump->p_scales + n * (Skp / 32), 0, (size_t)(Skp / 32));
      if (nk > 0) {
        double qh[256];
        q_hat(op, g, b, h, i, qh);
        double l = 0.0;
        float M = -INFINITY;
        int M_set = 0;
        float s[128];
        double pt[128], ds[128];                 /* ds: score uncertainty (ambiguity bound) */
        double* A = NULL;                        /* ambiguity accumulators, when asked for */
        double Bsum = 0.0, dM = 0.0;
        int undetermined = 0, jM = -1;           /* jM: key whose score set M */
        if (dump && dump->amb) {
          A = dump->amb + n * D;
          for (int d = 0; d < D; ++d) A[d] = 0.0;
        }
        for (int t = 0; t * BN < nk; ++t) {
          int j0 = t * BN, j1 = j0 + BN < nk ? j0 + BN : nk;   /* visible keys of this tile */
          ++tv;
          float mx = -INFINITY;
          int jmx = j0;
          for (int j = j0; j < j1; ++j) {
            double acc = 0.0, aabs = 0.0;
            for (int d0 = 0; d0 < D; d0 += 32) {
              double blk = 0.0;
              for (int d = d0; d < d0 + 32; ++d) blk += qh[d] * kv.kh[(int64_t)j * D + d];
              acc += blk;
              aabs += fabs(blk);
            }
            s[j - j0] = (dump && dump->s_in) ? dump->s_in[n * Skp + j] : (float)(acc * (1.0 + opt->s_perturb));
            /* given scores (a kernel's own) carry no score uncertainty */
            ds[j - j0] = (dump && dump->s_in) ? 0.0
                         : AMB_S * aabs + (opt->s_perturb != 0.0 ? fabs((double)s[j - j0] * opt->s_perturb) : 0.0);
            if (s[j - j0] > mx) { mx = s[j - j0]; jmx = j; }
          }
          float x = mx * c;
          /* uncertainty of x (fp32 product of an uncertain score); none when the scores
             are given: every later fp32 step is then the kernel's own, bit for bit */
          const double rt = (dump && dump->s_in) ? 0.0 : 1.2e-7;
          const double dx = (double)c * ds[jmx - j0] + rt * fabs((double)x);
          if (!M_set) {
            M = x;
            M_set = 1;
            dM = dx;
            jM = jmx;
          } else {
            const double thr = (double)(M + opt->delta);
            if (A && fabs((double)x - thr) <= dx + dM + rt * fabs(thr) && rt > 0.0) undetermined = 1;
            if (x > M + opt->delta) {
              float Mn = x;
              double alpha = exp2((double)(M - Mn));
              for (int d = 0; d < D; ++d) o[d] *= alpha;
              l *= alpha;
              if (A) {
                /* alpha itself is uncertain (M, M' and the kernel's exp2): everything
                   accumulated so far carries that relative error */
                const double ra = 0.6931471805599453 * (dM + dx) + AMB_X;
                for (int d = 0; d < D; ++d) A[d] = A[d] * alpha + ra * fabs(o[d]);
                Bsum = Bsum * alpha + ra * l;
              }
              M = Mn;
              dM = dx;
              jM = jmx;
              ++fb;
            }
          }
          if (dump && dump->m_frozen) dump->m_frozen[n * ntiles + t] = M;
          for (int jb = j0; jb < j1; jb += 32) {
            int je = jb + 32 < j1 ? jb + 32 : j1;
            float smax = -INFINITY;
            for (int j = jb; j < je; ++j) if (s[j - j0] > smax) smax = s[j - j0];
            float tmax = smax * c - M;       /* fp32(fp32(smax*c) - M): 0 in the block holding M */
            int E = (int)floorf(tmax + phi) - emax;
            if (E < -127) E = -127;
            if (E > 127) E = 127;
            float bE = M + (float)E;
            float Bk = opt->beta - opt->efq_a * bE;   /* EFQ: fp32(b - fp32(a bE)) */
            double sc = ldexp(1.0, E);
            int blk_undet = 0;
            if (A && smax != -INFINITY) {
              int jsm = jb;
              for (int j = jb; j < je; ++j) if (s[j - j0] == smax) { jsm = j; break; }
              /* the block holding the score that set M has tmax = 0 exactly on both sides */
              if (jM >= jb && jM < je && s[jM - j0] == smax) jsm = -1;
              if (jsm >= 0) {
                const double dt = (double)c * ds[jsm - j0] + dM + rt * (fabs((double)(smax * c)) + fabs((double)M));
                const double tp = (double)(tmax + phi);
                const int Elo = (int)floor(tp - dt), Ehi = (int)floor(tp + dt);
                if (Elo != Ehi && Ehi - emax > -127 && Elo - emax < 127) blk_undet = 1;
              }
            }
            for (int j = jb; j < je; ++j) {
              float r = fmaf(s[j - j0], c, -bE);
              uint32_t code;
              int hw = (opt->mufu_mask >> (j % 32)) & 1;
              uint32_t alt;
              if (efq) {
                float y = fmaf(s[j - j0], a_c, Bk);                 /* one rounding to fp32 */
                double kk = nearbyint((double)y);                 /* ties to even */
                if (!(kk > 0.0)) kk = 0.0;
                if (kk > 7.0) kk = 7.0;
                code = (uint32_t)kk;
                alt = code;
              } else {
                code = orc_encode(efmt, (double)exp2_model(r, hw, pc));
                alt = code;
                if (hw && dump && dump->p_alt) {
                  const uint32_t lo = orc_encode(efmt, exp2((double)r) * (1.0 - AMB_X));
                  const uint32_t hi = orc_encode(efmt, exp2((double)r) * (1.0 + AMB_X));
                  alt = code == lo ? hi : lo;
                }
              }
              if (dump && dump->p_alt) dump->p_alt[n * Skp + j] = (uint8_t)alt;
              const uint32_t used = (dump && dump->p_in) ? dump->p_in[n * Skp + j] : code;
              pt[j - j0] = orc_decode(efmt, used) * sc;
              if (A && s[j - j0] != -INFINITY && !(dump && dump->p_in)) {   /* given codes: determined */
                double dp = 0.0;
                if (blk_undet) {
                  /* requantised one exponent step finer or coarser */
                  dp = 0.25 * pt[j - j0] + orc_decode(efmt, 1) * sc * 2.0;
                } else {
                  const double dr = (double)c * ds[j - j0] + dM + rt * (fabs((double)s[j - j0] * c) + fabs((double)bE));
                  const double rlo = (double)r - dr, rhi = (double)r + dr;
                  uint32_t clo, chi;
                  if (efq) {
                    const double dy = (double)opt->efq_a * dr;
                    const double y = (double)fmaf(s[j - j0], a_c, Bk);
                    double klo = nearbyint(y - dy), khi = nearbyint(y + dy);
                    klo = klo < 0.0 ? 0.0 : (klo > 7.0 ? 7.0 : klo);
                    khi = khi < 0.0 ? 0.0 : (khi > 7.0 ? 7.0 : khi);
                    clo = (uint32_t)klo; chi = (uint32_t)khi;
                  } else if (hw) {
                    clo = orc_encode(efmt, exp2(rlo) * (1.0 - AMB_X));
                    chi = orc_encode(efmt, exp2(rhi) * (1.0 + AMB_X));
                  } else {
                    const double rp = rt > 0.0 ? 1e-7 : 0.0;   /* the cubic is bit-exact given the scores */
                    clo = orc_encode(efmt, (double)exp2_model((float)rlo, 0, pc) * (1.0 - rp));
                    chi = orc_encode(efmt, (double)exp2_model((float)rhi, 0, pc) * (1.0 + rp));
                  }
                  if (clo != chi) dp = fabs(orc_decode(efmt, chi) - orc_decode(efmt, clo)) * sc;
                }
                if (dp > 0.0) {
                  Bsum += dp;
                  for (int d = 0; d < D; ++d) A[d] += dp * fabs(kv.vh[(int64_t)d * kv.nk + j]);
                }
              }
              if (dump && dump->p_codes) dump->p_codes[n * Skp + j] = (uint8_t)code;
            }
            if (dump && dump->p_scales) dump->p_scales[n * (Skp / 32) + jb / 32] = (uint8_t)(E + 127);
          }
          if (dump && dump->s) for (int j = j0; j < j1; ++j) dump->s[n * Skp + j] = s[j - j0];
          for (int j = j0; j < j1; ++j) l += pt[j - j0];
          for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            const double* vr = kv.vh + (int64_t)d * kv.nk;
            for (int j = j0; j < j1; ++j) acc += pt[j - j0] * vr[j];
            o[d] += acc;
          }
        }
        for (int d = 0; d < D; ++d) o[d] = l > 0.0 ? o[d] / l : 0.0;
        if (A) {
          for (int d = 0; d < D; ++d) {
            const double den = l - Bsum;
            A[d] = undetermined ? INFINITY
                                : (Bsum == 0.0 ? 0.0 : (den > 0.0 ? (A[d] + Bsum * fabs(o[d])) / den : INFINITY));
          }
        }
      }
      if (fallbacks) fallbacks[n] = fb;
      if (tiles_visited) tiles_visited[n] = tv;
    }
    kv_free(&kv);
  }
  free(order); free(gstart);
}

/* ------------------------------------------------------------------------- */
/* O5-bf16: emulation of the exact-softmax BF16 baseline (standard attention  */
/* of the [FSA-digest] figure, tiled FlashAttention-style with the online row  */
/* maximum and historical rescaling that [EFQ] abstract keeps unchanged).       */
/* Per row over key tiles of 128: s_j = fp32(exact dot of bf16 q, k); first    */
/* tile M = fp32(mx*c); later x = fp32(mx*c), if fp32(x - M) > tau: rescale by  */
/* 2^(M - x), M = x (lazy rescale: P stays below 2^tau, exact in the end);      */
/* p_j = bf16_rn(2^fmaf(s_j, c, -M)); O_acc += p v, l += p; O = O_acc / l.      */
/* ------------------------------------------------------------------------- */
static double bf16_round(double x) {
  float f = (float)x;
  uint32_t u; memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;     /* ties to even; inputs are finite */
  memcpy(&f, &u, 4);
  return (double)f;
}

void orc_bf16_emulate(const uint16_t* q, const uint16_t* k, const uint16_t* v, const orc_geom* g, float scale,
                      float tau, const int64_t* rows, int64_t nrows, double* out, int32_t* rescales, int nthreads) {
  const int D = g->D, BN = 128;
  const float c = (float)((double)scale * 1.4426950408889634073599246810018921);
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  int64_t* gstart = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  int64_t ng = group_rows(g, rows, nrows, order, gstart);
  for (int64_t gi = 0; gi < ng; ++gi) {
    int b0, h0, i0, kvh0;
    row_coords(g, rows[order[gstart[gi]]], &b0, &h0, &i0, &kvh0);
    orc_kv kv;
    kv_from_bf16(k, v, g, b0, kvh0, group_nk(g, rows, order, gstart[gi], gstart[gi + 1]), &kv, nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t t0 = gstart[gi]; t0 < gstart[gi + 1]; ++t0) {
      int64_t n = order[t0];
      int b, h, i, kvh;
      row_coords(g, rows[n], &b, &h, &i, &kvh);
      int nk = last_visible(g, i) + 1;
      double* o = out + n * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      int nres = 0;
      if (nk > 0) {
        const uint16_t* qr = q + (((int64_t)b * g->H + h) * g->Sq + i) * D;
        double qd[256];
        for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(qr[d]);
        double l = 0.0;
        float M = -INFINITY;
        int M_set = 0;
        float s[128];
        for (int j0 = 0; j0 < nk; j0 += BN) {
          int j1 = j0 + BN < nk ? j0 + BN : nk;
          float mx = -INFINITY;
          for (int j = j0; j < j1; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qd[d] * kv.kh[(int64_t)j * D + d];
            s[j - j0] = (float)acc;
            if (s[j - j0] > mx) mx = s[j - j0];
          }
          float x = mx * c;
          if (!M_set) { M = x; M_set = 1; }
          else if (x - M > tau) {
            double alpha = exp2((double)(M - x));
            for (int d = 0; d < D; ++d) o[d] *= alpha;
            l *= alpha;
            M = x;
            ++nres;
          }
          for (int j = j0; j < j1; ++j) {
            double p = bf16_round((double)(float)exp2((double)fmaf(s[j - j0], c, -M)));
            l += p;
            const double* vr = kv.vh;
            for (int d = 0; d < D; ++d) o[d] += p * vr[(int64_t)d * kv.nk + j];
          }
        }
        for (int d = 0; d < D; ++d) o[d] = l > 0.0 ? o[d] / l : 0.0;
      }
      if (rescales) rescales[n] = nres;
    }
    kv_free(&kv);
  }
  free(order); free(gstart);
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

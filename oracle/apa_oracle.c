/*
 * apa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, FP64 CPU statement of adaptive-precision attention (APA) as
 * described in "APA: sloppy attention, exact where it counts" (rfriedmann.de
 * blog), with the GQA / tail-aligned causal semantics of the FFPA docs
 * (ffpa-attn.readthedocs.io, the "Note" on cross, GQA and causal attention).
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * may load this library.  It shares no code with the CUDA path.
 *
 * Notation (log2 units, as the kernels use them):
 *   G = Hq/Hkv; packed row p = pos*G + g of KV head h (query head h*G+g);
 *   16-row groups are 16 consecutive packed rows; key tiles are 64 keys;
 *   row at query position i sees key j iff j <= i + (Nkv - Nq) (causal).
 *
 * Floating-point conventions.  Every step the kernels do in FP32 and that must
 * be bit-exact (the NVFP4 quantizer, the key mean) is written here as an FP64
 * operation followed by rounding to FP32, f32(); for + - * / that is the
 * correctly rounded FP32 result, because 53 >= 2*24 + 2.  Everything else
 * (scores, softmax, the hot test, pass 2, the merge) is plain FP64.
 *
 * Parity pins (the functions' checks against things other than themselves)
 * live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define TILE 64
#define GROUP_ROWS 16
#define LOG2E 1.4426950408889634073599
#define LN2 0.6931471805599453094172

static double f32(double x) { return (double)(float)x; }

double oracle_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ---------------------------------------------------------------------------
 * NVFP4 element and scale formats (blog, "Pass 1: FP4 everywhere, with a hot
 * test"): E2M1 elements can hold 0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6;
 * one UE4M3 scale (max 448) per 16 values; one FP32 scale per head so that
 * the head maximum maps to 6 * 448 = 2688.
 * ------------------------------------------------------------------------- */

static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* E2M1 code of x, round to nearest with ties to the even code, saturating at
 * +-6.  The sign bit is kept, so a small negative value becomes code 8 (-0). */
int oracle_e2m1_code(double x) {
  int sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 8 : 0;
  double a = fabs(x);
  int c;
  /* Decision points are the midpoints of neighbouring values; at a midpoint
   * the even code (0, 2, 4, 6) wins. */
  if (a <= 0.25) c = 0;
  else if (a < 0.75) c = 1;
  else if (a <= 1.25) c = 2;
  else if (a < 1.75) c = 3;
  else if (a <= 2.5) c = 4;
  else if (a < 3.5) c = 5;
  else if (a <= 5.0) c = 6;
  else c = 7;
  return sign | c;
}

double oracle_e2m1_value(int code) {
  double m = E2M1_MAG[code & 7];
  return (code & 8) ? -m : m;
}

/* UE4M3 (unsigned E4M3, bias 7, 3 mantissa bits, subnormals, max 448) code of
 * x >= 0, round to nearest with ties to even, saturating at 448. */
int oracle_ue4m3_code(double x) {
  if (!(x > 0.0)) return 0;
  if (x >= 448.0) return 0x7E;
  if (x < 0.015625) { /* below the minimum normal 2^-6: subnormal spacing 2^-9 */
    double q = rint(x * 512.0); /* default rounding mode: ties to even */
    return (int)q;              /* q == 8 is the code of 2^-6 as well */
  }
  int e;
  double f = frexp(x, &e); /* x = f * 2^e, f in [0.5, 1) */
  double mant = rint((2.0 * f - 1.0) * 8.0);
  int E = e - 1 + 7;
  if (mant >= 8.0) { mant = 0.0; E += 1; }
  int code = (E << 3) | (int)mant;
  if (code > 0x7E) code = 0x7E;
  return code;
}

double oracle_ue4m3_value(int code) {
  int E = (code >> 3) & 15, m = code & 7;
  if (E == 0) return ldexp((double)m, -9);
  return ldexp(1.0 + m / 8.0, E - 7);
}

/* The FP32 per-head scale: the head's largest magnitude maps to 2688. */
double oracle_head_scale(double amax) {
  if (amax == 0.0) return 1.0;
  return f32(amax / 2688.0);
}

/* Quantizes nblk blocks of 16 FP32 values with head scale s.
 * Per block: a = max|x|; scale code sb = UE4M3(fp32(a / fp32(6 s)));
 * if sb == 0 every code is 0, else code = E2M1(fp32(x * fp32(1 / fp32(sb s)))).
 * Dequantized value = E2M1(code) * UE4M3(sb) * s. */
/* E2M1 codes of one block under scale code sb; returns the FP32 sum of squared
 * errors sum_i fp32(x_i - fp32(E2M1(code_i) * D))^2, accumulated in index order
 * with every product and sum rounded to FP32 (D = fp32(UE4M3(sb) * s)). */
static double block_codes(const float* xb, double s, int sb, uint8_t* codes) {
  double D = f32(oracle_ue4m3_value(sb) * s);
  double inv = f32(1.0 / D);
  double err = 0.0;
  for (int i = 0; i < 16; ++i) {
    codes[i] = (uint8_t)oracle_e2m1_code(f32((double)xb[i] * inv));
    double t = f32((double)xb[i] - f32(oracle_e2m1_value(codes[i]) * D));
    err = f32(err + f32(t * t));
  }
  return err;
}

/* lse != 0: least-squared-error block scales (the APA page, "Second hunt": every
 * block scale picked from a small set of candidates by least squared error
 * instead of the nearest one).  Reading taken: the candidates are the nearest
 * code sb and its neighbours sb - 1 and sb + 1 (within 1..126), tried in that
 * order; a candidate replaces the current pick only with a strictly smaller
 * error (block_codes).  An all-zero block keeps code 0. */
void oracle_quantize_blocks_mode(const float* x, int64_t nblk, double s, uint8_t* codes, uint8_t* sf, int lse) {
  for (int64_t b = 0; b < nblk; ++b) {
    const float* xb = x + b * 16;
    double a = 0.0;
    for (int i = 0; i < 16; ++i) a = fmax(a, fabs((double)xb[i]));
    double t = f32(6.0 * s);
    double r = f32(a / t);
    int sb = oracle_ue4m3_code(r);
    sf[b] = (uint8_t)sb;
    if (sb == 0) {
      for (int i = 0; i < 16; ++i) codes[b * 16 + i] = 0;
      continue;
    }
    double best = block_codes(xb, s, sb, codes + b * 16);
    if (!lse) continue;
    const int cand[2] = {sb - 1, sb + 1};
    for (int j = 0; j < 2; ++j) {
      if (cand[j] < 1 || cand[j] > 0x7E) continue;
      uint8_t c2[16];
      double e = block_codes(xb, s, cand[j], c2);
      if (e < best) {
        best = e;
        sf[b] = (uint8_t)cand[j];
        memcpy(codes + b * 16, c2, 16);
      }
    }
  }
}

void oracle_quantize_blocks(const float* x, int64_t nblk, double s, uint8_t* codes, uint8_t* sf) {
  oracle_quantize_blocks_mode(x, nblk, s, codes, sf, 0);
}

/* The FP4 residual of Q ("Second hunt": Q2 is the FP4 residual Q - Q1 in the
 * same scale).  Reading taken: the same FP32 per-head scale s, block scales of
 * their own, and the residual formed in FP32 in this order, per element:
 *   q1 = E2M1(code1) * UE4M3(sb1)   (exact: at most 7 significant bits)
 *   d1 = fp32(q1 * s),  r = fp32(x - d1);
 * then r is quantized like any other 16-value block with scale s. */
void oracle_quantize_residual_blocks(const float* x, int64_t nblk, double s, const uint8_t* codes1,
                                     const uint8_t* sf1, uint8_t* codes2, uint8_t* sf2, int lse) {
  float r[16];
  for (int64_t b = 0; b < nblk; ++b) {
    for (int i = 0; i < 16; ++i) {
      double q1 = oracle_e2m1_value(codes1[b * 16 + i]) * oracle_ue4m3_value(sf1[b]);
      double d1 = f32(q1 * s);
      r[i] = (float)f32((double)x[b * 16 + i] - d1);
    }
    oracle_quantize_blocks_mode(r, 1, s, codes2 + b * 16, sf2 + b, lse);
  }
}

/* Tiles per range of the key-mean sum. */
#define MEAN_RANGE_TILES 64

/* Per-channel key mean mu_c of one KV head (blog, "Mean-centred K").  The
 * rounding is pinned so that the kernels can reproduce it bit for bit:
 *   1. per 64-key tile, an FP32 sum over the tile's keys in ascending order;
 *   2. per range of 64 consecutive tiles, an FP64 sum of the tile sums in
 *      ascending order (starting from 0);
 *   3. the range sums added in ascending order in FP64;
 *   4. divided by Nkv in FP64 and rounded to FP32. */
void oracle_key_mean(const uint16_t* k, int Nkv, int d, float* mu) {
  int T = (Nkv + TILE - 1) / TILE;
  for (int c = 0; c < d; ++c) {
    double S = 0.0;
    for (int t0 = 0; t0 < T; t0 += MEAN_RANGE_TILES) {
      double Sr = 0.0;
      for (int t = t0; t < t0 + MEAN_RANGE_TILES && t < T; ++t) {
        double acc = 0.0;
        int j1 = (t + 1) * TILE < Nkv ? (t + 1) * TILE : Nkv;
        for (int j = t * TILE; j < j1; ++j) acc = f32(acc + oracle_bf16_to_double(k[(int64_t)j * d + c]));
        Sr += acc;
      }
      S += Sr;
    }
    mu[c] = (float)(S / (double)Nkv);
  }
}

/* ---------------------------------------------------------------------------
 * Online-softmax state merge (blog, "The merge that makes it exact"):
 *   M = max(m1, m2), w_i = 2^(m_i - M), O = (w1 o1 + w2 o2) / (w1 l1 + w2 l2)
 * in log2 units.  A state with m = -inf is empty and gets weight 0.
 * Returns log2 of the merged sum, M + log2(w1 l1 + w2 l2).
 * ------------------------------------------------------------------------- */
double oracle_merge(double m1, double l1, const double* o1, double m2, double l2, const double* o2,
                    int d, double* out) {
  double M = fmax(m1, m2);
  double w1 = isinf(m1) && m1 < 0 ? 0.0 : exp2(m1 - M);
  double w2 = isinf(m2) && m2 < 0 ? 0.0 : exp2(m2 - M);
  double L = w1 * l1 + w2 * l2;
  for (int c = 0; c < d; ++c) out[c] = (w1 * o1[c] + w2 * o2[c]) / L;
  return M + log2(L);
}

/* ---------------------------------------------------------------------------
 * Exact attention in FP64 from the bf16 inputs: the target the method
 * approximates.  softmax(q k^T / sqrt(d) + mask) v, and the natural-log LSE.
 * rows: optional list of (b, hq, pos) triples; NULL = every row.
 * ------------------------------------------------------------------------- */
void oracle_exact(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int Hq, int Hkv, int Nq,
                  int Nkv, int d, int causal, const int32_t* rows, int64_t nrows, double* out, double* lse) {
  int G = Hq / Hkv, off = Nkv - Nq;
  int64_t total = rows ? nrows : (int64_t)B * Hq * Nq;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)Nkv);
    double* qd = (double*)malloc(sizeof(double) * (size_t)d);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < total; ++r) {
      int b, h, i;
      if (rows) { b = rows[3 * r]; h = rows[3 * r + 1]; i = rows[3 * r + 2]; }
      else { b = (int)(r / ((int64_t)Hq * Nq)); h = (int)((r / Nq) % Hq); i = (int)(r % Nq); }
      int hk = h / G;
      const uint16_t* qr = q + (((int64_t)b * Hq + h) * Nq + i) * d;
      const uint16_t* kh = k + ((int64_t)b * Hkv + hk) * (int64_t)Nkv * d;
      const uint16_t* vh = v + ((int64_t)b * Hkv + hk) * (int64_t)Nkv * d;
      int nvis = causal ? i + off + 1 : Nkv;
      for (int c = 0; c < d; ++c) qd[c] = oracle_bf16_to_double(qr[c]);
      double mx = -INFINITY;
      for (int j = 0; j < nvis; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += qd[c] * oracle_bf16_to_double(kh[(int64_t)j * d + c]);
        s[j] = dot / sqrt((double)d);
        if (s[j] > mx) mx = s[j];
      }
      double L = 0.0;
      for (int c = 0; c < d; ++c) acc[c] = 0.0;
      for (int j = 0; j < nvis; ++j) {
        double p = exp(s[j] - mx);
        L += p;
        for (int c = 0; c < d; ++c) acc[c] += p * oracle_bf16_to_double(vh[(int64_t)j * d + c]);
      }
      int64_t orow = ((int64_t)b * Hq + h) * Nq + i;
      for (int c = 0; c < d; ++c) out[orow * d + c] = acc[c] / L;
      if (lse) lse[orow] = mx + log(L);
    }
    free(s); free(qd); free(acc);
  }
}

/* ---------------------------------------------------------------------------
 * APA emulation.
 *
 * Quantization switches (blog, "Second hunt: which operand is to blame": the
 * host emulation that applies one quantization at a time):
 *   bit 0 Q, bit 1 K, bit 2 V, bit 3 P.  With a bit clear that operand stays
 *   exact (FP64) in pass 1; with all four clear pass 1 is exact attention over
 *   the cold tiles and the result equals exact attention for any eps.
 * ------------------------------------------------------------------------- */
#define QUANT_Q 1
#define QUANT_K 2
#define QUANT_V 4
#define QUANT_P 8
#define QUANT_Q2 16 /* Q as two FP4 terms, Q1 + FP4(Q - Q1) ("Second hunt"); needs QUANT_Q */
#define QUANT_LSE 32 /* least-squared-error block scales for Q, K and V ("Second hunt") */
#define QUANT_VWEIGHT 64 /* value-norm-weighted hot test ("Honest limits"); not a quantization */

typedef struct {
  double eps;         /* hot-test threshold; 0 = every visible tile hot, +inf = none */
  double tau;         /* lazy-max threshold in log2 units ("Lazy maximum": 4) */
  double cold_offset; /* a hot tile lifts the frame only to max(m, c - offset) (32; 0 = APA 0.2.0) */
  int quant;          /* QUANT_* bits */
} oracle_apa_params;

/* NVFP4 codes of one KV head (blog, "Pass 1" and "Mean-centred K"):
 *   mu [d]            key mean (oracle_key_mean);
 *   kcodes [Nkv][d]   E2M1 codes of fp32(k - mu), 16 channels per scale;
 *   ksf [Nkv][d/16]   UE4M3 scale codes; *s_k the FP32 head scale;
 *   vcodes [d][Npad]  E2M1 codes of V^T, 16 keys per scale (Npad = Nkv rounded
 *                     up to 16, the missing keys quantized as 0);
 *   vsf [d][Npad/16]  UE4M3 scale codes; *s_v the FP32 head scale. */
void oracle_quantize_kv_head(const uint16_t* kh, const uint16_t* vh, int Nkv, int d, float* mu,
                             uint8_t* kcodes, uint8_t* ksf, double* s_k, uint8_t* vcodes, uint8_t* vsf,
                             double* s_v, int lse) {
  oracle_key_mean(kh, Nkv, d, mu);
  float* kc = (float*)malloc(sizeof(float) * (size_t)Nkv * d);
  double amax = 0.0;
  for (int64_t e = 0; e < (int64_t)Nkv * d; ++e) {
    kc[e] = (float)(oracle_bf16_to_double(kh[e]) - (double)mu[e % d]);
    amax = fmax(amax, fabs((double)kc[e]));
  }
  *s_k = oracle_head_scale(amax);
  oracle_quantize_blocks_mode(kc, (int64_t)Nkv * d / 16, *s_k, kcodes, ksf, lse);
  free(kc);
  int Npad = (Nkv + 15) / 16 * 16;
  amax = 0.0;
  for (int64_t e = 0; e < (int64_t)Nkv * d; ++e) amax = fmax(amax, fabs(oracle_bf16_to_double(vh[e])));
  *s_v = oracle_head_scale(amax);
  float* vt = (float*)malloc(sizeof(float) * (size_t)Npad);
  for (int c = 0; c < d; ++c) {
    for (int j = 0; j < Npad; ++j) vt[j] = j < Nkv ? (float)oracle_bf16_to_double(vh[(int64_t)j * d + c]) : 0.0f;
    oracle_quantize_blocks_mode(vt, Npad / 16, *s_v, vcodes + (int64_t)c * Npad, vsf + (int64_t)c * (Npad / 16), lse);
  }
  free(vt);
}

/* NVFP4 codes of one query head: codes [Nq][d], sf [Nq][d/16], *s_q; with
 * codes2 / sf2 non-null also the codes of the residual term (same layout). */
void oracle_quantize_q_head(const uint16_t* qh, int Nq, int d, uint8_t* codes, uint8_t* sf, double* s_q,
                            uint8_t* codes2, uint8_t* sf2, int lse) {
  float* x = (float*)malloc(sizeof(float) * (size_t)Nq * d);
  double amax = 0.0;
  for (int64_t e = 0; e < (int64_t)Nq * d; ++e) {
    x[e] = (float)oracle_bf16_to_double(qh[e]);
    amax = fmax(amax, fabs((double)x[e]));
  }
  *s_q = oracle_head_scale(amax);
  oracle_quantize_blocks_mode(x, (int64_t)Nq * d / 16, *s_q, codes, sf, lse);
  if (codes2 && sf2) oracle_quantize_residual_blocks(x, (int64_t)Nq * d / 16, *s_q, codes, sf, codes2, sf2, lse);
  free(x);
}

/* Per (b, KV head) operands of pass 1. */
typedef struct {
  int Nkv, d, T;
  double* kq;  /* [Nkv][d] pass-1 K (centred; dequantized without s_k when K is quantized) */
  double* vq;  /* [Nkv][d] pass-1 V (dequantized without s_v when V is quantized) */
  double s_k, s_v;
  float* mu;   /* [d] key mean */
  float* wv;   /* [T] value-norm weight of each tile (oracle_value_weights) */
} head_ops;

/* Value-norm weights of one KV head's tiles (the APA page, "Honest limits": the
 * hot test bounds a cold tile's share of the softmax mass, not of the output; a
 * test weighted by value norm would target the rows where they differ).  The
 * page gives no formula; reading taken, with every step rounded to FP32:
 *   n_j = sqrt(sum_c fp32(v_jc^2)), the sum in channel order;
 *   a_t = max of n_j over the tile's keys;
 *   nbar = mean of n_j over all keys: FP32 sums per tile in key order, FP64 sums
 *          of those per range of 64 tiles and of the ranges, / Nkv, to FP32
 *          (the key mean's order);
 *   w_t = a_t / nbar (1 if nbar is 0).
 * The weighted test is l_t * w_t * 2^(m~ - m) > eps * lambda; lambda stays the
 * plain mass. */
void oracle_value_weights(const uint16_t* vh, int Nkv, int d, float* w) {
  int T = (Nkv + TILE - 1) / TILE;
  float* amax = (float*)malloc(sizeof(float) * T);
  float* tsum = (float*)malloc(sizeof(float) * T);
  for (int t = 0; t < T; ++t) {
    double a = 0.0, sum = 0.0;
    int j1 = (t + 1) * TILE < Nkv ? (t + 1) * TILE : Nkv;
    for (int j = t * TILE; j < j1; ++j) {
      double acc = 0.0;
      for (int c = 0; c < d; ++c) {
        double x = oracle_bf16_to_double(vh[(int64_t)j * d + c]);
        acc = f32(acc + f32(x * x));
      }
      double n = f32(sqrt(acc));
      a = fmax(a, n);
      sum = f32(sum + n);
    }
    amax[t] = (float)a;
    tsum[t] = (float)sum;
  }
  double S = 0.0;
  for (int t0 = 0; t0 < T; t0 += MEAN_RANGE_TILES) {
    double Sr = 0.0;
    for (int t = t0; t < t0 + MEAN_RANGE_TILES && t < T; ++t) Sr += (double)tsum[t];
    S += Sr;
  }
  double nbar = f32(S / (double)Nkv);
  for (int t = 0; t < T; ++t) w[t] = nbar == 0.0 ? 1.0f : (float)f32((double)amax[t] / nbar);
  free(amax);
  free(tsum);
}

static void prepare_head(const uint16_t* kh, const uint16_t* vh, int Nkv, int d, int quant, head_ops* H) {
  int T = (Nkv + TILE - 1) / TILE, Npad = (Nkv + 15) / 16 * 16;
  H->Nkv = Nkv; H->d = d; H->T = T;
  H->wv = (float*)malloc(sizeof(float) * (size_t)T);
  oracle_value_weights(vh, Nkv, d, H->wv);
  H->kq = (double*)malloc(sizeof(double) * (size_t)Nkv * d);
  H->vq = (double*)malloc(sizeof(double) * (size_t)Nkv * d);
  H->mu = (float*)malloc(sizeof(float) * (size_t)d);
  uint8_t* kcodes = (uint8_t*)malloc((size_t)Nkv * d);
  uint8_t* ksf = (uint8_t*)malloc((size_t)Nkv * d / 16);
  uint8_t* vcodes = (uint8_t*)malloc((size_t)Npad * d);
  uint8_t* vsf = (uint8_t*)malloc((size_t)Npad * d / 16);
  double s_k, s_v;
  oracle_quantize_kv_head(kh, vh, Nkv, d, H->mu, kcodes, ksf, &s_k, vcodes, vsf, &s_v, (quant & QUANT_LSE) != 0);
  if (quant & QUANT_K) {
    H->s_k = s_k;
    for (int64_t e = 0; e < (int64_t)Nkv * d; ++e)
      H->kq[e] = oracle_e2m1_value(kcodes[e]) * oracle_ue4m3_value(ksf[e / 16]);
  } else {
    /* exact centred keys (not rounded to FP32) */
    H->s_k = 1.0;
    for (int64_t e = 0; e < (int64_t)Nkv * d; ++e)
      H->kq[e] = oracle_bf16_to_double(kh[e]) - (double)H->mu[e % d];
  }
  if (quant & QUANT_V) {
    H->s_v = s_v;
    for (int c = 0; c < d; ++c)
      for (int j = 0; j < Nkv; ++j)
        H->vq[(int64_t)j * d + c] = oracle_e2m1_value(vcodes[(int64_t)c * Npad + j]) *
                                    oracle_ue4m3_value(vsf[(int64_t)c * (Npad / 16) + j / 16]);
  } else {
    H->s_v = 1.0;
    for (int64_t e = 0; e < (int64_t)Nkv * d; ++e) H->vq[e] = oracle_bf16_to_double(vh[e]);
  }
  free(kcodes); free(ksf); free(vcodes); free(vsf);
}

static void free_head(head_ops* H) { free(H->kq); free(H->vq); free(H->mu); free(H->wv); }

/* Q of one query head: per-head scale over the whole (b, h) slice, 16 channels per scale. */
static double q_head_scale(const uint16_t* qh, int Nq, int d) {
  double amax = 0.0;
  for (int64_t e = 0; e < (int64_t)Nq * d; ++e) amax = fmax(amax, fabs(oracle_bf16_to_double(qh[e])));
  return oracle_head_scale(amax);
}

static void quantize_q_row(const uint16_t* qr, int d, double s_q, int quant, double* out) {
  if (!(quant & QUANT_Q)) {
    for (int c = 0; c < d; ++c) out[c] = oracle_bf16_to_double(qr[c]);
    return;
  }
  float x[16];
  uint8_t codes[16], sf, codes2[16], sf2;
  for (int b = 0; b < d / 16; ++b) {
    for (int i = 0; i < 16; ++i) x[i] = (float)oracle_bf16_to_double(qr[b * 16 + i]);
    const int lse = (quant & QUANT_LSE) != 0;
    oracle_quantize_blocks_mode(x, 1, s_q, codes, &sf, lse);
    for (int i = 0; i < 16; ++i) out[b * 16 + i] = oracle_e2m1_value(codes[i]) * oracle_ue4m3_value(sf);
    if (quant & QUANT_Q2) {  /* both terms in units of s_q, accumulated against the same K */
      oracle_quantize_residual_blocks(x, 1, s_q, codes, &sf, codes2, &sf2, lse);
      for (int i = 0; i < 16; ++i) out[b * 16 + i] += oracle_e2m1_value(codes2[i]) * oracle_ue4m3_value(sf2);
    }
  }
}

/* The clamp of the P group scale ("The bug: a sink that drowned the tail":
 * the scale exponent is clamped at -6, so the scale stays a normal UE4M3
 * value; 2^-6 is the smallest one). */
#define P_SCALE_MIN 0.015625

/* P of one row over one 64-key tile, encoded directly in FP4 (blog, "Pass 1:
 * FP4 everywhere, with a hot test", step 2: each 16-key group gets its own
 * scale, folded into the exponent bias; "Lazy maximum": tau = 4; "Second
 * hunt": the group scales are UE4M3, so each group maximum lands near 6; "The
 * bug": the scale exponent is clamped at -6).
 *   s[64]   the row's scores in log2 units, -inf where the key is not visible;
 *   m       the row's frame before this tile (-inf before its first tile);
 *   c       the tile maximum (out); mt the frame P is computed in (out):
 *           c if c > m + tau else m  (an empty tile keeps m);
 *   sc[4]   per 16-key group k: UE4M3_RN(2^(g_k - mt) / 6), at least 2^-6,
 *           g_k the group maximum (2^-6 for a group with nothing visible);
 *   p[64]   sc_k * E2M1_RN(2^(s - mt) / sc_k), 0 where masked; with quant_p = 0
 *           the exact 2^(s - mt) instead (the emulation's P switch).
 * Returns l_t, the sum of p in index order (the tile's FP4 row sum, step 3). */
double oracle_p_tile(const double* s, double m, double tau, int quant_p, double* c_out, double* mt_out,
                     double* sc, double* p) {
  double g[TILE / 16], c = -INFINITY;
  for (int kg = 0; kg < TILE / 16; ++kg) {
    g[kg] = -INFINITY;
    for (int jj = kg * 16; jj < kg * 16 + 16; ++jj)
      if (s[jj] > g[kg]) g[kg] = s[jj];
    c = fmax(c, g[kg]);
  }
  *c_out = c;
  if (c == -INFINITY) {
    *mt_out = m;
    for (int kg = 0; kg < TILE / 16; ++kg) sc[kg] = P_SCALE_MIN;
    for (int jj = 0; jj < TILE; ++jj) p[jj] = 0.0;
    return 0.0;
  }
  double mtl = (c > m + tau) ? c : m;
  *mt_out = mtl;
  double sum = 0.0;
  for (int kg = 0; kg < TILE / 16; ++kg) {
    double sck = P_SCALE_MIN;
    if (g[kg] != -INFINITY) {
      sck = oracle_ue4m3_value(oracle_ue4m3_code(exp2(g[kg] - mtl) / 6.0));
      if (sck < P_SCALE_MIN) sck = P_SCALE_MIN;
    }
    sc[kg] = sck;
    for (int jj = kg * 16; jj < kg * 16 + 16; ++jj) {
      double pj = 0.0;
      if (s[jj] != -INFINITY) {
        double x = exp2(s[jj] - mtl);
        pj = quant_p ? sck * oracle_e2m1_value(oracle_e2m1_code(x / sck)) : x;
      }
      p[jj] = pj;
      sum += pj;
    }
  }
  return sum;
}

/* Emulates pass 1, pass 2 and the merge for one 16-row group of one KV head.
 *
 * Pass 1 ("Pass 1: FP4 everywhere, with a hot test"), per tile in the order
 * tile 0, then from the group's causal diagonal backwards ("Tile order"):
 *   s    = (Q_fp4 . Kc_fp4) * s_q * s_k * log2(e) / sqrt(d), masked to -inf;
 *   g_k  = max of s over 16-key group k, c = max_k g_k;
 *   m~   = c if c > m + tau else m                       ("Lazy maximum");
 *   sc_k = UE4M3(2^(g_k - m~) / 6) clamped to >= 2^-6    (UE4M3 P scales,
 *          "Second hunt"; the clamp, "The bug");
 *   P    = sc_k * E2M1(2^(s - m~) / sc_k)                (P directly in FP4);
 *   l_t  = sum of P                                      (the ones-tile sum);
 *   hot  iff some row of the group has l_t * 2^(m~ - m) > eps * lambda, with
 *          lambda the running sum over the tiles judged before this one;
 *   hot:  m' = max(m, c - offset), lambda' = lambda 2^(m-m') + l_t 2^(m~-m'),
 *         l and o rescaled to m'                         (decoupled cold frame);
 *   cold: m' = m~, lambda, l, o rescaled to m', lambda += l_t, l += l_t,
 *         o += P . V_fp4.
 * Pass 2 ("Pass 2: exact FP16 on the hot tiles"): exact softmax over the keys
 * of the row's hot tiles with centred logits (q.k - q.mu) log2(e)/sqrt(d),
 * i.e. in the same frame as pass 1.
 * Merge ("The merge that makes it exact"), then the natural-log LSE with the
 * centring constant q.mu/sqrt(d) added back.
 *
 * diag_ell: optional [16][T]: l_t of each row expressed in the row's final
 *           frame (NaN where the row sees nothing of the tile).
 * diag_lam: optional [16]: final lambda (in the final frame).
 * diag_frame: optional [16][T][3]: per row and tile it sees, the tile maximum
 *           c, the frame m~ its P was computed in and the frame after the
 *           commit (NaN where the row sees nothing of the tile).
 */
static void apa_group(const uint16_t* q, const uint16_t* k, const uint16_t* v, int b, int hk, int grp,
                      int B, int Hq, int Hkv, int Nq, int Nkv, int d, int causal,
                      const oracle_apa_params* P, const head_ops* H, const double* s_q_heads,
                      double* out, double* lse, uint32_t* hot_mask, double* diag_ell, double* diag_lam,
                      double* diag_frame) {
  (void)B;
  int G = Hq / Hkv, R = G * Nq, T = H->T, off = Nkv - Nq;
  int nwords = (T + 31) / 32;
  int ngroups = (R + GROUP_ROWS - 1) / GROUP_ROWS;
  int p0 = grp * GROUP_ROWS;
  int nr = R - p0 < GROUP_ROWS ? R - p0 : GROUP_ROWS;
  double inv_sqrt_d = 1.0 / sqrt((double)d);
  const uint16_t* kh = k + ((int64_t)b * Hkv + hk) * (int64_t)Nkv * d;
  const uint16_t* vh = v + ((int64_t)b * Hkv + hk) * (int64_t)Nkv * d;

  double* qq = (double*)malloc(sizeof(double) * GROUP_ROWS * d);   /* pass-1 Q rows */
  double* qx = (double*)malloc(sizeof(double) * GROUP_ROWS * d);   /* exact Q rows */
  double* o = (double*)calloc((size_t)GROUP_ROWS * d, sizeof(double));
  double* hot_tile = (double*)calloc((size_t)T, sizeof(double)); /* 1.0 where the group is hot */
  double* ell = (double*)malloc(sizeof(double) * GROUP_ROWS * T);
  double* frame = (double*)malloc(sizeof(double) * GROUP_ROWS * T);
  double m[GROUP_ROWS], lam[GROUP_ROWS], l[GROUP_ROWS], cs[GROUP_ROWS];
  int pos[GROUP_ROWS], hq[GROUP_ROWS], lastv[GROUP_ROWS];
  double s[GROUP_ROWS][TILE], pv[GROUP_ROWS][TILE];
  double mt[GROUP_ROWS], lt[GROUP_ROWS], ct[GROUP_ROWS];
  int empty[GROUP_ROWS];

  int tmax = 0;
  for (int r = 0; r < nr; ++r) {
    int p = p0 + r;
    pos[r] = p / G;
    hq[r] = hk * G + p % G;
    const uint16_t* qr = q + (((int64_t)b * Hq + hq[r]) * Nq + pos[r]) * d;
    quantize_q_row(qr, d, s_q_heads[p % G], P->quant, qq + r * d);
    for (int c = 0; c < d; ++c) qx[r * d + c] = oracle_bf16_to_double(qr[c]);
    cs[r] = ((P->quant & QUANT_Q) ? s_q_heads[p % G] : 1.0) * H->s_k * LOG2E * inv_sqrt_d;
    lastv[r] = causal ? pos[r] + off : Nkv - 1;
    if (lastv[r] / TILE > tmax) tmax = lastv[r] / TILE;
    m[r] = -INFINITY; lam[r] = 0.0; l[r] = 0.0;
  }
  for (int e = 0; e < GROUP_ROWS * T; ++e) { ell[e] = NAN; frame[e] = NAN; }

  for (int step = 0; step <= tmax; ++step) {
    int t = step == 0 ? 0 : tmax + 1 - step; /* 0, tmax, tmax-1, ..., 1 */
    int j0 = t * TILE;
    /* scores, frame candidate, P and l_t per row */
    for (int r = 0; r < nr; ++r) {
      for (int jj = 0; jj < TILE; ++jj) {
        int j = j0 + jj;
        if (j >= Nkv || j > lastv[r]) { s[r][jj] = -INFINITY; continue; }
        double dot = 0.0;
        for (int ch = 0; ch < d; ++ch) dot += qq[r * d + ch] * H->kq[(int64_t)j * d + ch];
        s[r][jj] = dot * cs[r];
      }
      double sc[TILE / 16];
      lt[r] = oracle_p_tile(s[r], m[r], P->tau, (P->quant & QUANT_P) != 0, &ct[r], &mt[r], sc, pv[r]);
      empty[r] = (ct[r] == -INFINITY);
    }
    /* the hot test: one verdict for the group.  eps = 0 is the all-exact run:
     * every tile the group can see is hot, even one whose FP4 mass rounds to 0. */
    int hot = 0;
    if (!isinf(P->eps)) {
      for (int r = 0; r < nr; ++r) {
        if (empty[r]) continue;
        if (P->eps == 0.0) { hot = 1; continue; }
        double w = (P->quant & QUANT_VWEIGHT) ? (double)H->wv[t] : 1.0;
        if (m[r] == -INFINITY) { if (lt[r] * w > 0.0) hot = 1; continue; }
        if (lt[r] * w * exp2(mt[r] - m[r]) > P->eps * lam[r]) hot = 1;
      }
    }
    if (hot) hot_tile[t] = 1.0;
    /* commit */
    for (int r = 0; r < nr; ++r) {
      if (empty[r]) continue;
      ell[r * T + t] = lt[r];
      frame[r * T + t] = mt[r];
      double mn, c = ct[r];
      if (hot) {
        mn = fmax(m[r], c - P->cold_offset);
        double f = m[r] == -INFINITY ? 0.0 : exp2(m[r] - mn);
        lam[r] = lam[r] * f + lt[r] * exp2(mt[r] - mn);
        l[r] *= f;
        for (int ch = 0; ch < d; ++ch) o[r * d + ch] *= f;
      } else {
        mn = mt[r];
        double f = m[r] == -INFINITY ? 0.0 : exp2(m[r] - mn);
        lam[r] = lam[r] * f + lt[r];
        l[r] = l[r] * f + lt[r];
        for (int ch = 0; ch < d; ++ch) {
          double acc = o[r * d + ch] * f;
          for (int jj = 0; jj < TILE; ++jj)
            if (pv[r][jj] != 0.0) acc += pv[r][jj] * H->vq[(int64_t)(j0 + jj) * d + ch];
          o[r * d + ch] = acc;
        }
      }
      m[r] = mn;
      if (diag_frame) {
        double* fr = diag_frame + ((int64_t)r * T + t) * 3;
        fr[0] = c; fr[1] = mt[r]; fr[2] = mn;
      }
    }
  }

  /* hot mask bits of this group */
  if (hot_mask) {
    uint32_t* w = hot_mask + (((int64_t)b * Hkv + hk) * ngroups + grp) * nwords;
    for (int i = 0; i < nwords; ++i) w[i] = 0;
    for (int t = 0; t < T; ++t)
      if (hot_tile[t] != 0.0) w[t / 32] |= 1u << (t % 32);
  }

  /* pass 2 (exact, hot tiles only) and the merge, per row */
  double* sk = (double*)malloc(sizeof(double) * (size_t)Nkv);
  double* o2 = (double*)malloc(sizeof(double) * d);
  double* o1 = (double*)malloc(sizeof(double) * d);
  double* res = (double*)malloc(sizeof(double) * d);
  for (int r = 0; r < nr; ++r) {
    double qmu = 0.0;
    for (int ch = 0; ch < d; ++ch) qmu += qx[r * d + ch] * (double)H->mu[ch];
    double m2 = -INFINITY;
    int any = 0;
    for (int t = 0; t < T; ++t) {
      if (hot_tile[t] == 0.0) continue;
      for (int j = t * TILE; j < (t + 1) * TILE && j < Nkv && j <= lastv[r]; ++j) {
        double dot = 0.0;
        for (int ch = 0; ch < d; ++ch) dot += qx[r * d + ch] * oracle_bf16_to_double(kh[(int64_t)j * d + ch]);
        sk[j] = (dot - qmu) * LOG2E * inv_sqrt_d;
        if (sk[j] > m2) m2 = sk[j];
        any = 1;
      }
    }
    double l2 = 0.0;
    for (int ch = 0; ch < d; ++ch) o2[ch] = 0.0;
    if (any) {
      for (int t = 0; t < T; ++t) {
        if (hot_tile[t] == 0.0) continue;
        for (int j = t * TILE; j < (t + 1) * TILE && j < Nkv && j <= lastv[r]; ++j) {
          double p = exp2(sk[j] - m2);
          l2 += p;
          for (int ch = 0; ch < d; ++ch) o2[ch] += p * oracle_bf16_to_double(vh[(int64_t)j * d + ch]);
        }
      }
    }
    for (int ch = 0; ch < d; ++ch) o1[ch] = o[r * d + ch] * H->s_v;
    double lg = oracle_merge(l[r] > 0.0 ? m[r] : -INFINITY, l[r], o1, m2, l2, o2, d, res);
    int64_t orow = ((int64_t)b * Hq + hq[r]) * Nq + pos[r];
    for (int ch = 0; ch < d; ++ch) out[orow * d + ch] = res[ch];
    if (lse) lse[orow] = LN2 * lg + qmu * inv_sqrt_d;
    if (diag_ell)
      for (int t = 0; t < T; ++t)
        diag_ell[r * T + t] = isnan(ell[r * T + t]) ? NAN : ell[r * T + t] * exp2(frame[r * T + t] - m[r]);
    if (diag_lam) diag_lam[r] = lam[r];
  }
  free(sk); free(o2); free(o1); free(res);
  free(qq); free(qx); free(o); free(hot_tile); free(ell); free(frame);
}

/* Runs the APA emulation over a list of 16-row groups.
 * units: optional [nunits][3] (b, hkv, group); NULL = every group.
 * out [B,Hq,Nq,d], lse [B,Hq,Nq]: written for the rows of the listed groups.
 * hot_mask [B,Hkv,ceil(R/16),ceil(T/32)]: written for the listed groups.
 * diag_ell [nunits][16][T], diag_lam [nunits][16], diag_frame [nunits][16][T][3]:
 * optional diagnostics (see apa_group).
 * Returns 0, or -1 on an unsupported shape. */
int oracle_apa(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int Hq, int Hkv, int Nq,
               int Nkv, int d, int causal, double eps, double tau, double cold_offset, int quant,
               const int32_t* units, int64_t nunits, double* out, double* lse, uint32_t* hot_mask,
               double* diag_ell, double* diag_lam, double* diag_frame) {
  if (Hq % Hkv || Nkv < Nq || d % 64 || Nq <= 0) return -1;
  oracle_apa_params P = {eps, tau, cold_offset, quant};
  int G = Hq / Hkv, R = G * Nq, T = (Nkv + TILE - 1) / TILE;
  int ngroups = (R + GROUP_ROWS - 1) / GROUP_ROWS;
  int64_t nu = units ? nunits : (int64_t)B * Hkv * ngroups;
  int32_t* all = NULL;
  if (!units) {
    all = (int32_t*)malloc(sizeof(int32_t) * 3 * (size_t)nu);
    for (int64_t u = 0; u < nu; ++u) {
      all[3 * u] = (int32_t)(u / ((int64_t)Hkv * ngroups));
      all[3 * u + 1] = (int32_t)((u / ngroups) % Hkv);
      all[3 * u + 2] = (int32_t)(u % ngroups);
    }
    units = all;
  }
  /* one (b, hkv) head at a time: its K/V operands are shared by its groups */
  char* done = (char*)calloc((size_t)nu, 1);
  double* sq = (double*)malloc(sizeof(double) * G);
  for (int64_t u0 = 0; u0 < nu; ++u0) {
    if (done[u0]) continue;
    int b = units[3 * u0], hk = units[3 * u0 + 1];
    head_ops H;
    prepare_head(k + ((int64_t)b * Hkv + hk) * (int64_t)Nkv * d, v + ((int64_t)b * Hkv + hk) * (int64_t)Nkv * d,
                 Nkv, d, quant, &H);
    for (int g = 0; g < G; ++g)
      sq[g] = q_head_scale(q + ((int64_t)b * Hq + hk * G + g) * (int64_t)Nq * d, Nq, d);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = u0; u < nu; ++u) {
      if (done[u] || units[3 * u] != b || units[3 * u + 1] != hk) continue;
      done[u] = 1;
      apa_group(q, k, v, b, hk, units[3 * u + 2], B, Hq, Hkv, Nq, Nkv, d, causal, &P, &H, sq, out, lse,
                hot_mask, diag_ell ? diag_ell + u * GROUP_ROWS * T : NULL,
                diag_lam ? diag_lam + u * GROUP_ROWS : NULL,
                diag_frame ? diag_frame + u * GROUP_ROWS * T * 3 : NULL);
    }
    free_head(&H);
  }
  free(sq); free(done); free(all);
  return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * csa2_oracle.c -- CPU oracle for the CSA2 long-context attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (libcsa2, its Python
 * binding) may link, load or call this file.  It is used by tests/, by the
 * smoke check in __graft_entry__.py and by the cpu_baseline / reference arm
 * of bench.py, and by nothing else.  It shares no source with the CUDA path.
 *
 * It is deliberately plain and slow: every step follows the definition on the
 * source pages, in the pages' order, with no blocking, fusion or reordering.
 * Floating point that the pages leave open is done in fp64 and rounded once.
 * Compile with -O2 -fno-fast-math -ffp-contract=off (no silent FMA contraction;
 * fmaf() is called where the definition below says FMA).
 *
 * Page names used in the citations:
 *   [P1] "DeepSeek V4.1 Flash 아키텍처 분석" (plaidlabs.ai blog)
 *   [P2] "DeepSeek Multi-Head Latent Attention(MLA) 해부" (huny.dev blog)
 *   [P3] "DeepSeek V4.1 Flash 해부, KV 캐시는 줄고 사후학습 레시피는 그대로" (traillabs.ai)
 *   [P4] "매개변수는 커졌는데 메모리는 4분의 1, DeepSeek V4.1 Flash의 KV 캐시 다이어트" (ithotfix.com)
 *   [P5] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence" (issue #58 translation)
 *
 * Readings of the pages taken here (where they are silent) are marked READING.
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_LAT 512  /* latent dims of a main-KV entry, [P1] "890 bytes/token은 어떻게 나오는가" */
#define ORC_ROPE 64  /* decoupled RoPE dims, [P2] §3 Decoupled RoPE (d_r = 64) */
#define ORC_DQK 576  /* ORC_LAT + ORC_ROPE: the score dimension of an absorbed query */
#define ORC_DI 128   /* indexer head dimension c_I, [P5] §4.2.1 */
#define ORC_WIN 128  /* sliding window n_win, [P5] §4.2.1 */

/* ------------------------------------------------------------------------ */
/* C1. Element formats.  [P1] "890 bytes/token": main KV = E2M1 data with an */
/* E4M3 scale per 16 values; indexer K = MXFP4 (E2M1 with an E8M0 scale per  */
/* 32).  [P4] "890이 맞아떨어지는 계산": FP4 max with a per-16 scale 448*6.   */
/* The codecs are the standard OCP definitions.                              */
/* ------------------------------------------------------------------------ */

/* E2M1: 1 sign bit (bit 3), 2 exponent bits (bias 1), 1 mantissa bit. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_decode(uint8_t code) {
  double m = E2M1_MAG[code & 7];
  return (code & 8) ? -m : m;
}

/* Round-to-nearest, ties to the even code, saturating at 6; the sign bit is
 * the input's sign bit (so a negative value that rounds to zero gives 0x8). */
uint8_t orc_e2m1_encode(float x) {
  double a = fabs((double)x);
  int best = 7;
  if (!(a > 6.0)) {
    best = 0;
    for (int c = 1; c < 8; ++c) {
      double dc = fabs(a - E2M1_MAG[c]);
      double db = fabs(a - E2M1_MAG[best]);
      if (dc < db || (dc == db && (c & 1) == 0)) best = c;
    }
  }
  return (uint8_t)(best | (signbit(x) ? 8 : 0));
}

/* E4M3 ("FN" variant): bias 7, no infinities, 0x7F/0xFF are NaN, max 448,
 * subnormals m * 2^-9. */
double orc_e4m3_decode(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Round-to-nearest, ties to even code, saturating at 448 (satfinite). */
uint8_t orc_e4m3_encode(float x) {
  double a = fabs((double)x);
  int best = 0x7E; /* 448 */
  if (!(a > 448.0)) {
    best = 0;
    for (int c = 1; c <= 0x7E; ++c) {
      double dc = fabs(a - orc_e4m3_decode((uint8_t)c));
      double db = fabs(a - orc_e4m3_decode((uint8_t)best));
      if (dc < db || (dc == db && (c & 1) == 0)) best = c;
    }
  }
  return (uint8_t)(best | (signbit(x) ? 0x80 : 0));
}

/* E8M0: 2^(code-127); 0xFF is NaN. */
double orc_e8m0_decode(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* bf16 round-to-nearest-even of an fp32 value (returns the 16-bit pattern). */
uint16_t orc_bf16_encode(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if (isnan(x)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lo = u & 0xFFFF0000u, hi = lo + 0x10000u; /* the two bf16 neighbours (same sign) */
  float flo, fhi;
  memcpy(&flo, &lo, 4);
  memcpy(&fhi, &hi, 4);
  double dlo = fabs((double)x - (double)flo), dhi = fabs((double)fhi - (double)x);
  if (isinf(fhi)) dhi = INFINITY;
  uint32_t pick;
  if (dlo < dhi) pick = lo;
  else if (dhi < dlo) pick = hi;
  else pick = ((lo >> 16) & 1) ? hi : lo; /* tie: even mantissa */
  return (uint16_t)(pick >> 16);
}

double orc_bf16_decode(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ------------------------------------------------------------------------ */
/* C3. Group quantisers.                                                     */
/* ------------------------------------------------------------------------ */

/* NVFP4-style group of 16 (main latent and RoPE sidecar).
 * [P1] "890 bytes/token": one 1-byte E4M3 scale per 16 values.
 * READING (the pages give the format, not the scale rule):
 *   s = E4M3(amax / 6) (IEEE fp32 division, RNE, satfinite);
 *   s == 0 -> all codes 0 and scale code 0;
 *   code_i = E2M1(x_i / s) with s the decoded scale (IEEE fp32 division).
 * Packing: byte j = code(2j) | code(2j+1) << 4. */
void orc_nvfp4_quant16(const float *x, uint8_t *codes8, uint8_t *scale) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  uint8_t sc = orc_e4m3_encode(amax / 6.0f);
  float s = (float)orc_e4m3_decode(sc);
  *scale = sc;
  for (int j = 0; j < 8; ++j) {
    uint8_t c0 = 0, c1 = 0;
    if (s != 0.0f) {
      c0 = orc_e2m1_encode(x[2 * j] / s);
      c1 = orc_e2m1_encode(x[2 * j + 1] / s);
    }
    codes8[j] = (uint8_t)(c0 | (c1 << 4));
  }
  if (s == 0.0f) *scale = 0;
}

/* floor(log2(a)) for a finite a > 0, read exactly from the representation. */
static int orc_floor_log2(float a) {
  int ex;
  (void)frexpf(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
  return ex - 1;
}

/* MXFP4 group of 32 (indexer keys and indexer queries), OCP MX rule:
 * e = floor(log2(amax)) - 2 (2 = emax of E2M1), clamped to [-127, 127];
 * scale code e + 127; amax == 0 -> scale code 0 and zero codes;
 * code_i = E2M1(x_i * 2^-e). */
void orc_mxfp4_quant32(const float *x, uint8_t *codes16, uint8_t *scale) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) {
    *scale = 0;
    memset(codes16, 0, 16);
    return;
  }
  int e = orc_floor_log2(amax) - 2;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  *scale = (uint8_t)(e + 127);
  for (int j = 0; j < 16; ++j) {
    uint8_t c0 = orc_e2m1_encode(ldexpf(x[2 * j], -e));
    uint8_t c1 = orc_e2m1_encode(ldexpf(x[2 * j + 1], -e));
    codes16[j] = (uint8_t)(c0 | (c1 << 4));
  }
}

/* MXFP8 group of 32 for the 8-bit sliding-window cache.
 * [P1] "890 bytes/token" and [P3]: the window KV stays in 8 bits ("FP8").
 * READING: E4M3 elements with one E8M0 scale per 32 values,
 * e = floor(log2(amax)) - 8 (8 = emax of E4M3); code_i = E4M3(x_i * 2^-e). */
void orc_mxfp8_quant32(const float *x, uint8_t *codes32, uint8_t *scale) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) {
    *scale = 0;
    memset(codes32, 0, 32);
    return;
  }
  int e = orc_floor_log2(amax) - 8;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  *scale = (uint8_t)(e + 127);
  for (int i = 0; i < 32; ++i) codes32[i] = orc_e4m3_encode(ldexpf(x[i], -e));
}

/* ------------------------------------------------------------------------ */
/* C9. RoPE on the last 64 dims ([P5] §2.3.3 "Partial Rotary Positional      */
/* Embedding"; [P2] §3 decoupled RoPE key of 64 dims).                       */
/* READING: interleaved pairs (2i, 2i+1), inv_freq_i = theta^(-2i/64),       */
/* angle = pos * inv_freq_i; cos/sin evaluated in double, rounded to fp32;   */
/* x' = fma(x, c, -(y*s)), y' = fma(y, c, x*s) with the products rounded.    */
/* ------------------------------------------------------------------------ */
void orc_rope_cs(double theta, int64_t pos, float *cs /* [32][2] */) {
  for (int i = 0; i < ORC_ROPE / 2; ++i) {
    double inv_freq = pow(theta, -(double)(2 * i) / (double)ORC_ROPE);
    double ang = (double)pos * inv_freq;
    cs[2 * i] = (float)cos(ang);
    cs[2 * i + 1] = (float)sin(ang);
  }
}

void orc_rope_apply(float *x64, const float *cs) {
  for (int i = 0; i < ORC_ROPE / 2; ++i) {
    float x = x64[2 * i], y = x64[2 * i + 1];
    float c = cs[2 * i], s = cs[2 * i + 1];
    float ys = y * s, xs = x * s;
    x64[2 * i] = fmaf(x, c, -ys);
    x64[2 * i + 1] = fmaf(y, c, xs);
  }
}

/* ------------------------------------------------------------------------ */
/* Entry encoding.  Quantisation happens after RoPE ([P4] "890이 맞아떨어지는 */
/* 계산").  The 512 latent dims form the pages' 288 B record; the 64 RoPE     */
/* dims are a 36 B sidecar in the same format (READING: the MLA split of [P2] */
/* keeps the RoPE key outside the 512-dim latent).                           */
/*   v[576] = entry vector in fp32, rope dims 512..575 NOT yet rotated        */
/*   ik[128] = indexer key                                                   */
/* Outputs: lat_codes[256], lat_scales[32], rope_codes[32], rope_scales[4],   */
/*          idx_codes[64], idx_scales[4].                                    */
/* ------------------------------------------------------------------------ */
void orc_encode_entry(const float *v, const float *ik, const float *cs, uint8_t *lat_codes,
                      uint8_t *lat_scales, uint8_t *rope_codes, uint8_t *rope_scales,
                      uint8_t *idx_codes, uint8_t *idx_scales) {
  float r[ORC_ROPE];
  memcpy(r, v + ORC_LAT, sizeof(r));
  orc_rope_apply(r, cs);
  for (int g = 0; g < ORC_LAT / 16; ++g) orc_nvfp4_quant16(v + 16 * g, lat_codes + 8 * g, lat_scales + g);
  for (int g = 0; g < ORC_ROPE / 16; ++g) orc_nvfp4_quant16(r + 16 * g, rope_codes + 8 * g, rope_scales + g);
  for (int b = 0; b < ORC_DI / 32; ++b) orc_mxfp4_quant32(ik + 32 * b, idx_codes + 16 * b, idx_scales + b);
}

/* The V4 entry, kept for comparison ([P5] §2.3.4: the KV entries are stored in
 * FP8 except the RoPE dims, which stay BF16).  READING: the FP8 part uses the
 * 8-bit window's MXFP8 rule (E4M3 with one E8M0 per 32 values); the RoPE dims
 * are rotated first, as for the V4.1 record.
 *   v[576] = entry vector, rope dims 512..575 NOT yet rotated; ik[128] = key
 * Outputs: lat_codes[512] (E4M3), lat_scales[16] (E8M0), rope_codes[128]
 *          (64 bf16, little-endian), idx_codes[64], idx_scales[4] (MXFP4). */
void orc_encode_entry_v4(const float *v, const float *ik, const float *cs, uint8_t *lat_codes,
                         uint8_t *lat_scales, uint8_t *rope_codes, uint8_t *idx_codes, uint8_t *idx_scales) {
  float r[ORC_ROPE];
  memcpy(r, v + ORC_LAT, sizeof(r));
  orc_rope_apply(r, cs);
  for (int b = 0; b < ORC_LAT / 32; ++b) orc_mxfp8_quant32(v + 32 * b, lat_codes + 32 * b, lat_scales + b);
  uint16_t *h = (uint16_t *)rope_codes;
  for (int i = 0; i < ORC_ROPE; ++i) h[i] = orc_bf16_encode(r[i]);
  for (int b = 0; b < ORC_DI / 32; ++b) orc_mxfp4_quant32(ik + 32 * b, idx_codes + 16 * b, idx_scales + b);
}

/* The indexer-key records alone of n entries (the idx planes of
 * orc_encode_entry, entry by entry): ik [n][128] -> idx_codes [n][64],
 * idx_scales [n][4].  Entries are independent, so rows run in parallel. */
void orc_encode_keys(int64_t n, const float *ik, uint8_t *idx_codes, uint8_t *idx_scales) {
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < n; ++e)
    for (int b = 0; b < ORC_DI / 32; ++b)
      orc_mxfp4_quant32(ik + e * ORC_DI + 32 * b, idx_codes + e * 64 + 16 * b, idx_scales + e * 4 + b);
}

/* One sliding-window slot from a token vector v[576] (rope dims not yet
 * rotated): rotate, then store 8-bit (MXFP8: 576 codes + 18 scales) or bf16. */
void orc_encode_swa(const float *v, const float *cs, int swa_mxfp8, uint8_t *codes /*576 or 1152 B*/,
                    uint8_t *scales /*18 B, MXFP8 only*/) {
  float t[ORC_DQK];
  memcpy(t, v, sizeof(t));
  orc_rope_apply(t + ORC_LAT, cs);
  if (swa_mxfp8) {
    for (int b = 0; b < ORC_DQK / 32; ++b) orc_mxfp8_quant32(t + 32 * b, codes + 32 * b, scales + b);
  } else {
    uint16_t *h = (uint16_t *)codes;
    for (int i = 0; i < ORC_DQK; ++i) h[i] = orc_bf16_encode(t[i]);
  }
}

/* ------------------------------------------------------------------------ */
/* C10. Overlapping token compression, ratio m ([P5] §2.3.1 "압축된          */
/* Key-Value Entry"): for each channel, a softmax over the 2m rows           */
/* [Z^a_{mi..m(i+1)-1} + B^a ; Z^b_{m(i-1)..mi-1} + B^b], then               */
/* C_i = sum S^a (.) C^a + sum S^b (.) C^b.  For i == 0 the b rows are       */
/* Z = -inf and C = 0.  Computed in fp64, rounded once to fp32.              */
/*   a_rows[r], b_rows[r] for r < m point at token rows of width `dim`       */
/*   (b_rows == NULL for i == 0); ba, bb are [m][dim].                       */
/* ------------------------------------------------------------------------ */
void orc_compress(int m, int dim, const float *const *ca_rows, const float *const *za_rows,
                  const float *const *cb_rows, const float *const *zb_rows, const float *ba,
                  const float *bb, float *out) {
  double logit[8], e[8];
  for (int j = 0; j < dim; ++j) {
    int n = 0;
    for (int r = 0; r < m; ++r) logit[n++] = (double)za_rows[r][j] + (double)ba[r * dim + j];
    for (int r = 0; r < m; ++r)
      logit[n++] = cb_rows ? (double)zb_rows[r][j] + (double)bb[r * dim + j] : -INFINITY;
    double mx = -INFINITY;
    for (int r = 0; r < 2 * m; ++r)
      if (logit[r] > mx) mx = logit[r];
    double den = 0.0;
    for (int r = 0; r < 2 * m; ++r) {
      e[r] = exp(logit[r] - mx);
      den += e[r];
    }
    double acc = 0.0;
    for (int r = 0; r < m; ++r) acc += (e[r] / den) * (double)ca_rows[r][j];
    for (int r = 0; r < m; ++r) {
      double c = cb_rows ? (double)cb_rows[r][j] : 0.0;
      acc += (e[m + r] / den) * c;
    }
    out[j] = (float)acc;
  }
}

/* ------------------------------------------------------------------------ */
/* C4. Lightning-indexer score ([P5] §2.3.1 "Sparse Selection을 위한         */
/* Lightning Indexer"):  I_{t,s} = sum_h w_{t,h} * ReLU(q_{t,h} . K_s),      */
/* with the indexer QK product in FP4 ([P5] §2.3.4): q_{t,h} is quantised to */
/* MXFP4 (groups of 32) and the dot is taken over the dequantised vectors.   */
/* READING: d_h = RN_fp32(exact dot); r_h = d_h > 0 ? d_h : +0;              */
/*   acc = +0; for h in order: acc = fma(w_h, r_h, acc).                     */
/* Returns flags: 1 if an fp64 partial sum could have been inexact (block    */
/* exponent span too wide), 2 if some d_h was not exactly representable in   */
/* fp32 (so a tensor-core accumulation need not reproduce it).               */
/* ------------------------------------------------------------------------ */
void orc_quant_q_index(int H, const uint16_t *q_bf16, uint8_t *q_codes /*H*64*/, uint8_t *q_scales /*H*4*/) {
  float tmp[ORC_DI];
  for (int h = 0; h < H; ++h) {
    for (int i = 0; i < ORC_DI; ++i) tmp[i] = (float)orc_bf16_decode(q_bf16[h * ORC_DI + i]);
    for (int b = 0; b < ORC_DI / 32; ++b)
      orc_mxfp4_quant32(tmp + 32 * b, q_codes + h * 64 + 16 * b, q_scales + h * 4 + b);
  }
}

static double orc_mxfp4_value(const uint8_t *codes, const uint8_t *scales, int i) {
  uint8_t byte = codes[i >> 1];
  uint8_t c = (i & 1) ? (byte >> 4) : (byte & 15);
  return orc_e2m1_decode(c) * orc_e8m0_decode(scales[i >> 5]);
}

int orc_index_score_rows(int64_t n, const uint8_t *idx_codes, const uint8_t *idx_scales,
                         const int64_t *rows, int H, const uint16_t *q_bf16, const float *w,
                         float *out) {
  int flags = 0;
  uint8_t *qc = (uint8_t *)malloc((size_t)H * 64);
  uint8_t *qs = (uint8_t *)malloc((size_t)H * 4);
  double *qv = (double *)malloc(sizeof(double) * (size_t)H * ORC_DI);
  orc_quant_q_index(H, q_bf16, qc, qs);
  for (int h = 0; h < H; ++h)
    for (int i = 0; i < ORC_DI; ++i) qv[h * ORC_DI + i] = orc_mxfp4_value(qc + h * 64, qs + h * 4, i);
  /* rows are independent: OpenMP over them only */
#pragma omp parallel for schedule(static) reduction(| : flags)
  for (int64_t t = 0; t < n; ++t) {
    int64_t s = rows ? rows[t] : t;
    const uint8_t *kc = idx_codes + s * 64, *ks = idx_scales + s * 4;
    double kv[ORC_DI];
    for (int i = 0; i < ORC_DI; ++i) kv[i] = orc_mxfp4_value(kc, ks, i);
    float acc = 0.0f;
    for (int h = 0; h < H; ++h) {
      /* exactness of the fp64 sum: all products are multiples of
       * 2^(eq+ek-2) and below 2^(eq+ek+6); 128 of them need < 53 bits of span */
      int emin = 1000, emax = -1000;
      for (int b = 0; b < ORC_DI / 32; ++b) {
        if (qs[h * 4 + b] == 0 || ks[b] == 0) continue; /* all-zero group */
        int e = (int)qs[h * 4 + b] + (int)ks[b] - 254;
        if (e < emin) emin = e;
        if (e > emax) emax = e;
      }
      if (emax > emin + 30) flags |= 1;
      double d = 0.0;
      for (int i = 0; i < ORC_DI; ++i) d += qv[h * ORC_DI + i] * kv[i];
      float df = (float)d;
      if ((double)df != d) flags |= 2;
      float r = df > 0.0f ? df : 0.0f;
      acc = fmaf(w[h], r, acc);
    }
    out[t] = acc;
  }
  free(qc);
  free(qs);
  free(qv);
  return flags;
}

/* ------------------------------------------------------------------------ */
/* C6. Top-k selector ([P5] §2.3.1: C^Sprs = {C_s | I_{t,s} in Top-k}).      */
/* Order: score descending, then position ascending (ties -> lower index);   */
/* -0 and +0 compare equal.  Output: the chosen positions in ascending       */
/* order, padded with -1.  Returns -1 on a NaN score.                        */
/* ------------------------------------------------------------------------ */
typedef struct {
  float score;
  int64_t pos;
} orc_item;

static int orc_item_cmp(const void *pa, const void *pb) {
  const orc_item *a = (const orc_item *)pa, *b = (const orc_item *)pb;
  if (a->score > b->score) return -1;
  if (a->score < b->score) return 1;
  if (a->pos < b->pos) return -1;
  if (a->pos > b->pos) return 1;
  return 0;
}

static int orc_i64_cmp(const void *pa, const void *pb) {
  int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
  return (a > b) - (a < b);
}

int orc_topk(int64_t n, const float *score, const int64_t *pos, int k, int32_t *out) {
  orc_item *it = (orc_item *)malloc(sizeof(orc_item) * (size_t)(n > 0 ? n : 1));
  for (int64_t i = 0; i < n; ++i) {
    if (isnan(score[i])) {
      free(it);
      return -1;
    }
    it[i].score = score[i];
    it[i].pos = pos ? pos[i] : i;
  }
  qsort(it, (size_t)n, sizeof(orc_item), orc_item_cmp);
  int64_t take = n < k ? n : k;
  int64_t *sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)(take > 0 ? take : 1));
  for (int64_t i = 0; i < take; ++i) sel[i] = it[i].pos;
  qsort(sel, (size_t)take, sizeof(int64_t), orc_i64_cmp);
  for (int i = 0; i < k; ++i) out[i] = i < take ? (int32_t)sel[i] : -1;
  free(sel);
  free(it);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* C7. Candidate pool of the Hierarchical Sparse Indexer ([P1] "512개를 고르기 */
/* 위해 매번 전체를 검색한다면"; [P4] "40개 층 중 바이트를 쓰는 곳은 넷"):     */
/* positions are grouped 8 at a time, a block's score is the max over its     */
/* positions, and at most 2,048 blocks are kept.                             */
/* READING: blocks are 8-aligned from position 0; only visible positions      */
/* (0..T-1) count; order (block max desc, block id asc); output ascending.   */
/* ------------------------------------------------------------------------ */
int orc_pool(int64_t T, const float *score, int block_size, int max_blocks, int32_t *pool_out,
             int32_t *count) {
  int64_t nb = (T + block_size - 1) / block_size;
  float *bm = (float *)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
  for (int64_t b = 0; b < nb; ++b) {
    float m = -INFINITY;
    for (int64_t p = b * block_size; p < (b + 1) * block_size && p < T; ++p) {
      if (isnan(score[p])) {
        free(bm);
        return -1;
      }
      if (score[p] > m) m = score[p];
    }
    bm[b] = m;
  }
  int rc = orc_topk(nb, bm, NULL, max_blocks, pool_out);
  *count = (int32_t)(nb < max_blocks ? nb : max_blocks);
  free(bm);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* C8. Core attention over the selected entries plus the window, fp64.       */
/* Shared-KV MQA ([P5] §2.3.1 "Shared Key-Value MQA"): each selected entry    */
/* is key and value.  Absorbed query form ([P2] §4): the logit is            */
/* q_lat . c + q_rope . k_rope, the value is the 512-dim latent c.           */
/* Window branch ([P5] §2.3.3 "Sliding Window Attention의 추가 Branch") and  */
/* sink ([P5] §2.3.3 "Attention Sink"): exp(z'_h) joins the denominator.     */
/*   z_j = sm_scale * (q . e_j) over 576 dims                                */
/*   o = sum_j exp(z_j - M) c_j[0:512] / (sum_j exp(z_j - M) + exp(z'_h - M)) */
/*   lse = M + log(denominator)                                               */
/* Entries: idx[0..k) (values < 0 skipped) from the FP4 cache, then n_swa    */
/* window slots (MXFP8: 576 codes + 18 scales, or bf16).                     */
/* Duplicates are kept as separate terms.                                    */
/* ------------------------------------------------------------------------ */
static void orc_dequant_nvfp4(const uint8_t *codes, const uint8_t *scales, int n, double *out) {
  for (int i = 0; i < n; ++i) {
    uint8_t byte = codes[i >> 1];
    uint8_t c = (i & 1) ? (byte >> 4) : (byte & 15);
    out[i] = orc_e2m1_decode(c) * orc_e4m3_decode(scales[i >> 4]);
  }
}

void orc_dequant_main(const uint8_t *lat_codes, const uint8_t *lat_scales, const uint8_t *rope_codes,
                      const uint8_t *rope_scales, double *out576) {
  orc_dequant_nvfp4(lat_codes, lat_scales, ORC_LAT, out576);
  orc_dequant_nvfp4(rope_codes, rope_scales, ORC_ROPE, out576 + ORC_LAT);
}

/* A V4 entry (orc_encode_entry_v4) back to 576 exact values. */
void orc_dequant_main_v4(const uint8_t *lat_codes, const uint8_t *lat_scales, const uint8_t *rope_codes,
                         double *out576) {
  for (int i = 0; i < ORC_LAT; ++i) out576[i] = orc_e4m3_decode(lat_codes[i]) * orc_e8m0_decode(lat_scales[i >> 5]);
  const uint16_t *h = (const uint16_t *)rope_codes;
  for (int i = 0; i < ORC_ROPE; ++i) out576[ORC_LAT + i] = orc_bf16_decode(h[i]);
}

void orc_dequant_swa(const uint8_t *codes, const uint8_t *scales, int swa_mxfp8, double *out576) {
  if (swa_mxfp8) {
    for (int i = 0; i < ORC_DQK; ++i) out576[i] = orc_e4m3_decode(codes[i]) * orc_e8m0_decode(scales[i >> 5]);
  } else {
    const uint16_t *h = (const uint16_t *)codes;
    for (int i = 0; i < ORC_DQK; ++i) out576[i] = orc_bf16_decode(h[i]);
  }
}

int orc_sparse_attn(int H, const uint16_t *q_bf16 /* H x 576 */, const uint8_t *lat_codes,
                    const uint8_t *lat_scales, const uint8_t *rope_codes, const uint8_t *rope_scales,
                    const int32_t *idx, int k, const uint8_t *swa_codes, int64_t swa_code_stride,
                    const uint8_t *swa_scales, int64_t swa_scale_stride, int n_swa, int swa_mxfp8,
                    const float *sink, float sm_scale, float *out /* H x 512 */, float *lse /* H */,
                    int entry_format /* 0: V4.1 FP4 record, 1: V4 FP8 + bf16 RoPE */) {
  int n = 0;
  for (int j = 0; j < k; ++j)
    if (idx[j] >= 0) ++n;
  n += n_swa;
  double *ent = (double *)malloc(sizeof(double) * ORC_DQK * (size_t)(n > 0 ? n : 1));
  int e = 0;
  for (int j = 0; j < k; ++j) {
    int64_t s = idx[j];
    if (s < 0) continue;
    if (entry_format == 1)
      orc_dequant_main_v4(lat_codes + s * 512, lat_scales + s * 16, rope_codes + s * 128, ent + (size_t)e * ORC_DQK);
    else
      orc_dequant_main(lat_codes + s * 256, lat_scales + s * 32, rope_codes + s * 32, rope_scales + s * 4,
                       ent + (size_t)e * ORC_DQK);
    ++e;
  }
  for (int j = 0; j < n_swa; ++j) {
    orc_dequant_swa(swa_codes + (int64_t)j * swa_code_stride,
                    swa_scales ? swa_scales + (int64_t)j * swa_scale_stride : NULL, swa_mxfp8,
                    ent + (size_t)e * ORC_DQK);
    ++e;
  }
  /* heads are independent: OpenMP over them only */
#pragma omp parallel for schedule(static)
  for (int h = 0; h < H; ++h) {
    double qd[ORC_DQK];
    double *z = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < ORC_DQK; ++i) qd[i] = orc_bf16_decode(q_bf16[h * ORC_DQK + i]);
    double M = -INFINITY;
    for (int j = 0; j < n; ++j) {
      double dot = 0.0;
      for (int i = 0; i < ORC_DQK; ++i) dot += qd[i] * ent[(size_t)j * ORC_DQK + i];
      z[j] = (double)sm_scale * dot;
      if (z[j] > M) M = z[j];
    }
    if (sink && (double)sink[h] > M) M = (double)sink[h];
    if (n == 0 && !sink) {
      for (int d = 0; d < ORC_LAT; ++d) out[h * ORC_LAT + d] = 0.0f;
      lse[h] = -INFINITY;
      free(z);
      continue;
    }
    double den = sink ? exp((double)sink[h] - M) : 0.0;
    for (int j = 0; j < n; ++j) {
      z[j] = exp(z[j] - M); /* z now holds the unnormalised weight */
      den += z[j];
    }
    for (int d = 0; d < ORC_LAT; ++d) {
      double acc = 0.0;
      for (int j = 0; j < n; ++j) acc += z[j] * ent[(size_t)j * ORC_DQK + d];
      out[h * ORC_LAT + d] = (float)(acc / den);
    }
    lse[h] = (float)(M + log(den));
    free(z);
  }
  free(ent);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Byte accounting (C2): the pages' per-entry and per-token sizes.           */
/* [P1] "890 bytes/token": 288 = 512*0.5 + 32; 68 = 64 + 4; 356 per entry;    */
/* per input token (3 encoder caches at 2 tokens/entry + 1 decoder cache).    */
/* ------------------------------------------------------------------------ */
int orc_main_entry_bytes(int dims, int group) { return dims / 2 + dims / group; }
int orc_mx_entry_bytes(int dims, int group) { return dims / 2 + dims / group; }

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads the parallel loops over independent rows use from now on (the
 * single-thread time of the CPU baseline); n <= 0 leaves the count as it is. */
void orc_set_num_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
}

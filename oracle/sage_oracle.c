/*
 * sage_oracle.c -- CPU oracle for SageAttention3's microscaled FP4 attention
 * forward.  TEST INFRASTRUCTURE ONLY (tests, smoke check, bench CPU baseline).
 *
 * Written from the method's description, step by step, in the order the
 * pages give it; see sage_oracle.h for the sources and the layouts.  Where the
 * pages are silent the plainest reading is taken and stated beside the code.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math), so
 * that every float operation below is a single IEEE round-to-nearest-even op.
 */
#include "sage_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Codecs.                                                                   */
/* ------------------------------------------------------------------------ */

/* E2M1 (FP4): bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa.
 * Exponent 0 is subnormal (0 or 0.5).  Eight magnitudes, sixteen codes, and
 * +0/-0 share a value: the 15 representable values of [NEWS-OBST]. */
double sor_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* Round to the nearest E2M1 value; a tie goes to the even code (mantissa bit
 * 0); magnitudes above 6 saturate to 6; the sign is kept, so a negative value
 * that rounds to zero is -0 (code 0x8).  The pages fix none of these: the
 * reading is IEEE-style nearest-even with saturation to the largest finite
 * value.  Implemented as a scan over the eight magnitudes. */
int sor_e2m1_encode(float x) {
  int sign = signbit(x) ? 8 : 0;
  double a = fabs((double)x);
  if (isnan(x)) return sign | 7;
  if (a >= 6.0) return sign | 7;
  int best = 0;
  double bestd = a;
  for (int i = 1; i < 8; i++) {
    double d = fabs(sor_e2m1_value(i) - a);
    if (d < bestd || (d == bestd && (i & 1) == 0)) {
      bestd = d;
      best = i;
    }
  }
  return sign | best;
}

/* E4M3 (FP8, the "FN" variant: no infinities, 0x7F/0xFF are NaN, largest
 * finite 448, consistent with the 448*6 of [NEWS-OBST]).  Exponent bias 7;
 * exponent field 0 is subnormal with step 2^-9. */
double sor_e4m3_value(int b) {
  int s = b & 0x80, E = (b >> 3) & 15, m = b & 7;
  if (E == 15 && m == 7) return NAN;
  double v = (E == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), E - 10);
  return s ? -v : v;
}

/* Round to nearest E4M3, ties to even, saturating to +-448. */
int sor_e4m3_encode(float x) {
  int sign = signbit(x) ? 0x80 : 0;
  double a = fabs((double)x);
  if (isnan(x) || a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal step 2^-9; rint() rounds half to even; 8 steps = 2^-6 is the
     * smallest normal, whose code is also 8 */
    return sign | (int)rint(a * 512.0);
  }
  int e;
  double f = frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) */
  double mant = (2.0 * f - 1.0) * 8.0; /* a = (1 + mant/8) * 2^(e-1) */
  int k = (int)rint(mant);
  int E = e - 1 + 7;
  if (k == 8) {
    k = 0;
    E += 1;
  }
  if (E > 15 || (E == 15 && k == 7)) return sign | 0x7E;
  return sign | (E << 3) | k;
}

static float f32_from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

void sor_encode_range(uint32_t first, uint32_t count, uint8_t *e2m1, uint8_t *e4m3) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)count; i++) {
    float x = f32_from_bits(first + (uint32_t)i);
    if (e2m1) e2m1[i] = (uint8_t)sor_e2m1_encode(x);
    if (e4m3) e4m3[i] = (uint8_t)sor_e4m3_encode(x);
  }
}

/* ------------------------------------------------------------------------ */
/* 1x16 NVFP4 group quantizer ([NEWS-OBST] 1x16 groups; [NEWS-HW] NVFP4).    */
/* ------------------------------------------------------------------------ */

/* scale = E4M3(amax / 6) so that the group's largest magnitude maps onto the
 * largest E2M1 value 6; codes = E2M1(x * (1/scale)).  Silent in the pages and
 * read here as: float division amax/6 rounded to nearest, the scale rounded
 * to nearest E4M3, the reciprocal 1/scale rounded to nearest float, one
 * rounded float product per element.  A zero scale (all-zero group, or
 * amax/6 below half the smallest E4M3 subnormal) gives all-zero codes. */
void sor_quant_group16(const float *x, uint8_t *codes16, uint8_t *scale) {
  float amax = 0.0f;
  for (int i = 0; i < 16; i++) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float q = amax / 6.0f;
  int sb = sor_e4m3_encode(q);
  float s = (float)sor_e4m3_value(sb);
  *scale = (uint8_t)sb;
  if (s == 0.0f) {
    for (int i = 0; i < 16; i++) codes16[i] = 0;
    return;
  }
  float r = 1.0f / s;
  for (int i = 0; i < 16; i++) {
    float y = x[i] * r;
    codes16[i] = (uint8_t)sor_e2m1_encode(y);
  }
}

static float bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

/* ------------------------------------------------------------------------ */
/* 1x32 MXFP4 group quantizer: the alternative the pages weighed and set     */
/* aside ([NEWS-HW]: E2M1 codes, 1x32 blocks, E8M0 scales).                  */
/* ------------------------------------------------------------------------ */

/* E8M0: an unsigned power-of-two exponent with bias 127; 0xFF is NaN. */
double sor_e8m0_value(int b) {
  if ((b & 0xFF) == 0xFF) return NAN;
  return ldexp(1.0, (b & 0xFF) - 127);
}

/* The pages give the format, not the rule.  The rule read here is the one the
 * OCP Microscaling (MX) v1.0 specification defines for MX conversion: the
 * shared exponent is floor(log2(amax)) minus the element format's largest
 * exponent (2 for E2M1), clamped to E8M0's range, and each element is
 * x / 2^shared rounded to nearest E2M1 (ties to even, saturating at 6).  The
 * division by a power of two is exact (ldexpf).  An all-zero group takes the
 * smallest scale byte and all-zero codes. */
void sor_quant_group32_mx(const float *x, uint8_t *codes32, uint8_t *scale) {
  float amax = 0.0f;
  for (int i = 0; i < 32; i++) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) {
    *scale = 0;
    for (int i = 0; i < 32; i++) codes32[i] = (uint8_t)sor_e2m1_encode(x[i]);
    return;
  }
  int E;
  frexpf(amax, &E); /* amax = f * 2^E, f in [0.5, 1): floor(log2(amax)) = E - 1 */
  int shared = (E - 1) - 2;
  if (shared < -127) shared = -127;
  if (shared > 127) shared = 127;
  *scale = (uint8_t)(shared + 127);
  for (int i = 0; i < 32; i++) codes32[i] = (uint8_t)sor_e2m1_encode(ldexpf(x[i], -shared));
}

/* One group of either format: NVFP4 (16 elements, E4M3 scale) or MXFP4 (32
 * elements, E8M0 scale). */
static void quant_group(int fmt, const float *x, uint8_t *codes, uint8_t *scale) {
  if (fmt == SOR_FMT_MXFP4)
    sor_quant_group32_mx(x, codes, scale);
  else
    sor_quant_group16(x, codes, scale);
}

static int group_size(int fmt) { return fmt == SOR_FMT_MXFP4 ? 32 : 16; }



static int round_up(int x, int m) { return (x + m - 1) / m * m; }

static void put_nibble(uint8_t *row, int idx, int code) {
  if (idx & 1)
    row[idx >> 1] = (uint8_t)((row[idx >> 1] & 0x0F) | (code << 4));
  else
    row[idx >> 1] = (uint8_t)((row[idx >> 1] & 0xF0) | (code & 0x0F));
}

static int get_nibble(const uint8_t *row, int idx) {
  return (idx & 1) ? (row[idx >> 1] >> 4) : (row[idx >> 1] & 0x0F);
}

/* Q and K: groups of consecutive elements along D, the contraction axis of
 * QK^T ([NEWS-OBST], solution 1): 16 for NVFP4, 32 for MXFP4.  No smoothing
 * (mean subtraction) of K: the pages do not describe one. */
void sor_quantize_rows_fmt(const uint16_t *x, int BH, int N, int D, int fmt, uint8_t *codes,
                           uint8_t *scales) {
  const int G = group_size(fmt);
  int N_pad = round_up(N, 128);
  size_t crow = (size_t)D / 2, srow = (size_t)D / G;
  memset(codes, 0, (size_t)BH * N_pad * crow);
  memset(scales, 0, (size_t)BH * N_pad * srow);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < (int64_t)BH * N; r++) {
    int64_t bh = r / N, n = r % N;
    const uint16_t *src = x + (size_t)r * D;
    uint8_t *cdst = codes + ((size_t)bh * N_pad + n) * crow;
    uint8_t *sdst = scales + ((size_t)bh * N_pad + n) * srow;
    for (int g = 0; g < D / G; g++) {
      float buf[32];
      uint8_t c[32];
      for (int i = 0; i < G; i++) buf[i] = bf16_to_f32(src[g * G + i]);
      quant_group(fmt, buf, c, &sdst[g]);
      for (int i = 0; i < G; i++) put_nibble(cdst, g * G + i, c[i]);
    }
  }
}

void sor_quantize_rows(const uint16_t *x, int BH, int N, int D, uint8_t *codes, uint8_t *scales) {
  sor_quantize_rows_fmt(x, BH, N, D, SOR_FMT_NVFP4, codes, scales);
}

/* V: the contraction axis of PV is the token axis, so the groups run along
 * tokens for each channel (block scales of a block-scaled product always run
 * along the contraction axis).  Output is V^T.  Tokens past N are zero, which
 * makes an all-padding NVFP4 group's scale and codes zero (an all-padding
 * MXFP4 group gets the smallest scale byte and zero codes). */
void sor_quantize_v_fmt(const uint16_t *v, int BH, int N, int D, int fmt, uint8_t *codes,
                        uint8_t *scales) {
  const int G = group_size(fmt);
  int N_pad = round_up(N, 128);
  size_t crow = (size_t)N_pad / 2, srow = (size_t)N_pad / G;
  memset(codes, 0, (size_t)BH * D * crow);
  memset(scales, 0, (size_t)BH * D * srow);
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t bh = 0; bh < BH; bh++) {
    for (int d = 0; d < D; d++) {
      uint8_t *cdst = codes + ((size_t)bh * D + d) * crow;
      uint8_t *sdst = scales + ((size_t)bh * D + d) * srow;
      for (int g = 0; g < N_pad / G; g++) {
        float buf[32];
        uint8_t c[32];
        for (int i = 0; i < G; i++) {
          int n = g * G + i;
          buf[i] = (n < N) ? bf16_to_f32(v[((size_t)bh * N + n) * D + d]) : 0.0f;
        }
        quant_group(fmt, buf, c, &sdst[g]);
        for (int i = 0; i < G; i++) put_nibble(cdst, g * G + i, c[i]);
      }
    }
  }
}

void sor_quantize_v(const uint16_t *v, int BH, int N, int D, uint8_t *codes, uint8_t *scales) {
  sor_quantize_v_fmt(v, BH, N, D, SOR_FMT_NVFP4, codes, scales);
}

/* ------------------------------------------------------------------------ */
/* Tiled attention with online softmax and two-level P quantization.         */
/* ------------------------------------------------------------------------ */

/* Decoding tables: the value of every E2M1 code and E4M3 byte, taken from the
 * codec definitions above. */
static double g_e2m1[16];
static double g_e4m3[256];
static double g_e8m0[256];
static int g_tables_ready = 0;

static void init_tables(void) {
  if (g_tables_ready) return;
#pragma omp critical(sor_tables)
  {
    if (!g_tables_ready) {
      for (int i = 0; i < 16; i++) g_e2m1[i] = sor_e2m1_value(i);
      for (int i = 0; i < 256; i++) g_e4m3[i] = sor_e4m3_value(i);
      for (int i = 0; i < 256; i++) g_e8m0[i] = sor_e8m0_value(i);
      g_tables_ready = 1;
    }
  }
}

#define SOR_MAX_D 256
#define SOR_MAX_TILE 512

/* One query row.  Softmax scale `scale` (the pages give none; callers pass
 * 1/sqrt(D), the standard one, unless they ask for another); below,
 * "/sqrt(D)" stands for "* scale".  Per KV tile, in ascending order:
 *   S_j    = sum_g sQ_g * sK_jg * sum_{k in g} q_k * k_jk   (decoded, exact)
 *   masked keys (j >= N, or j > i when causal) get S = -inf
 *   t      = max_j S_j over the tile, m_new = max(m_old, t)
 *   l      = l * exp((m_old - m_new)/sqrt(D)) + sum_j exp((S_j - m_new)/sqrt(D))
 *            (l is built from the unquantized probabilities)
 *   level 1 (TILE):    P2_j = 2688 * exp((S_j - t)/sqrt(D)),  sP1 = exp((t - m_new)/sqrt(D)) / 2688
 *           (RUNNING): P2_j = 2688 * exp((S_j - m_new)/sqrt(D)), sP1 = 1/2688
 *            -- the per-token first level that brings each token's values
 *            into [0, 448*6] ([NEWS-OBST], solution 2); P2_j is rounded to float.
 *   level 2: the group quantizer on P2 along keys (16 consecutive elements
 *            of a row, [NEWS-HW]; 32 for MXFP4)
 * For MXFP4 (fmt 1) every group is 32 elements with an E8M0 scale, and the
 * level-1 target 2688 = 448*6 (largest E4M3 scale times largest E2M1 value,
 * the range level 1 exists to fill) becomes 6: an E8M0 scale needs no help
 * with its range, and 6 keeps each row's tile maximum exactly representable
 * (scale 2^0, code 6), as 2688 does for NVFP4 (scale 448, code 6).
 *   acc    = acc * exp((m_old - m_new)/sqrt(D)) + sP1 * sum_j dec(P2_j) * dec(V_j)
 * and finally O = acc / l.
 * lnorm 1 (Direct-P, the rit.work summary of "Hardware-Aware FP4
 * FlashAttention-4", "Что сделали"): the normaliser is summed from the same
 * rounded probabilities that enter PV, sP1 * dec(P2_j) for each key, instead
 * of the unquantized exp((S_j - m_new)/sqrt(D)); the page defines no other
 * arithmetic, so the codes are still those of level 2 above. */
static void attend_row(const uint8_t *qc, const uint8_t *qs, const uint8_t *kc, const uint8_t *ks,
                       const uint8_t *vc, const uint8_t *vs, int N, int N_pad, int D, int causal,
                       int fmt, double scale, int pmode, int lnorm, int kv_tile, int i, double *out,
                       double *out_l, double *out_m) {
  const double isd = scale;
  const int GS = group_size(fmt);                            /* elements per scale */
  const int G = D / GS;                                      /* Q/K groups per row */
  const double *sc = (fmt == SOR_FMT_MXFP4) ? g_e8m0 : g_e4m3; /* scale values */
  const double R = (fmt == SOR_FMT_MXFP4) ? 6.0 : 2688.0;     /* level-1 target */
  double qv[SOR_MAX_D];
  double acc[SOR_MAX_D];
  double S[SOR_MAX_TILE];
  float P2[SOR_MAX_TILE];
  uint8_t pc[SOR_MAX_TILE];
  uint8_t ps[SOR_MAX_TILE / 16];

  const uint8_t *qrow = qc + (size_t)i * (D / 2);
  for (int d = 0; d < D; d++) qv[d] = g_e2m1[get_nibble(qrow, d)];
  for (int d = 0; d < D; d++) acc[d] = 0.0;
  double m = -INFINITY, l = 0.0;

  int kend = causal ? (i + 1) : N; /* keys j < kend are visible */
  for (int j0 = 0; j0 < kend; j0 += kv_tile) {
    int T = kv_tile;
    /* S for the tile */
    double t = -INFINITY;
    for (int jj = 0; jj < T; jj++) {
      int j = j0 + jj;
      if (j >= N || j >= kend) {
        S[jj] = -INFINITY;
        continue;
      }
      const uint8_t *krow = kc + (size_t)j * (D / 2);
      double s = 0.0;
      for (int g = 0; g < G; g++) {
        double part = 0.0;
        for (int k = GS * g; k < GS * g + GS; k++) part += qv[k] * g_e2m1[get_nibble(krow, k)];
        s += sc[qs[(size_t)i * G + g]] * sc[ks[(size_t)j * G + g]] * part;
      }
      S[jj] = s;
      if (s > t) t = s;
    }
    double m_new = (t > m) ? t : m;
    double alpha = exp((m - m_new) * isd);
    double lt = 0.0;
    for (int jj = 0; jj < T; jj++) lt += exp((S[jj] - m_new) * isd);

    /* level 1 */
    double ref = (pmode == 0) ? t : m_new;
    double sP1 = (pmode == 0) ? exp((t - m_new) * isd) / R : 1.0 / R;
    for (int jj = 0; jj < T; jj++) P2[jj] = (float)(R * exp((S[jj] - ref) * isd));
    /* level 2 */
    for (int g = 0; g < T / GS; g++) quant_group(fmt, &P2[GS * g], &pc[GS * g], &ps[g]);

    if (lnorm == 1) {
      /* Direct-P: the tile's share of l from the rounded probabilities */
      double rounded = 0.0;
      for (int g = 0; g < T / GS; g++) {
        double part = 0.0;
        for (int k = 0; k < GS; k++) part += g_e2m1[pc[GS * g + k]];
        rounded += sc[ps[g]] * part;
      }
      lt = sP1 * rounded;
    }
    l = l * alpha + lt;

    /* O update */
    for (int d = 0; d < D; d++) {
      const uint8_t *vrow = vc + (size_t)d * (N_pad / 2);
      const uint8_t *vsrow = vs + (size_t)d * (N_pad / GS);
      double pv = 0.0;
      for (int g = 0; g < T / GS; g++) {
        int jg = (j0 / GS) + g; /* token group index */
        if (GS * jg >= N_pad) break;
        double part = 0.0;
        for (int k = 0; k < GS; k++)
          part += g_e2m1[pc[GS * g + k]] * g_e2m1[get_nibble(vrow, GS * jg + k)];
        pv += sc[ps[g]] * sc[vsrow[jg]] * part;
      }
      acc[d] = acc[d] * alpha + sP1 * pv;
    }
    m = m_new;
  }
  for (int d = 0; d < D; d++) out[d] = acc[d] / l;
  if (out_l) *out_l = l;
  if (out_m) *out_m = m;
}

int sor_attention_ex(const uint8_t *qc, const uint8_t *qs, const uint8_t *kc, const uint8_t *ks,
                     const uint8_t *vc, const uint8_t *vs, int BH, int N, int D, int causal,
                     int fmt, double scale, int pmode, int lnorm, int kv_tile, const int64_t *rows,
                     int64_t nrows, double *out, double *out_l, double *out_m) {
  if (fmt != SOR_FMT_NVFP4 && fmt != SOR_FMT_MXFP4) return -1;
  if (lnorm != 0 && lnorm != 1) return -1;
  const int GS = group_size(fmt);
  if (D % GS || D > SOR_MAX_D || kv_tile % GS || kv_tile > SOR_MAX_TILE || kv_tile <= 0 || N < 1 ||
      !(scale > 0.0) || isinf(scale))
    return -1;
  init_tables();
  int N_pad = round_up(N, 128);
  int64_t total = rows ? nrows : (int64_t)BH * N;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < total; r++) {
    int64_t id = rows ? rows[r] : r;
    int64_t bh = id / N;
    int i = (int)(id % N);
    attend_row(qc + (size_t)bh * N_pad * (D / 2), qs + (size_t)bh * N_pad * (D / GS),
               kc + (size_t)bh * N_pad * (D / 2), ks + (size_t)bh * N_pad * (D / GS),
               vc + (size_t)bh * D * (N_pad / 2), vs + (size_t)bh * D * (N_pad / GS), N, N_pad, D,
               causal, fmt, scale, pmode, lnorm, kv_tile, i, out + (size_t)r * D, out_l ? out_l + r : 0,
               out_m ? out_m + r : 0);
  }
  return 0;
}

int sor_attention(const uint8_t *qc, const uint8_t *qs, const uint8_t *kc, const uint8_t *ks,
                  const uint8_t *vc, const uint8_t *vs, int BH, int N, int D, int causal,
                  int fmt, double scale, int pmode, int kv_tile, const int64_t *rows,
                  int64_t nrows, double *out, double *out_l, double *out_m) {
  return sor_attention_ex(qc, qs, kc, ks, vc, vs, BH, N, D, causal, fmt, scale, pmode, 0, kv_tile,
                          rows, nrows, out, out_l, out_m);
}

/* Exact softmax(scale * Q K^T) V in double, from the bf16 inputs. */
int sor_attention_exact(const uint16_t *q, const uint16_t *k, const uint16_t *v, int BH, int N,
                        int D, int causal, double scale, const int64_t *rows, int64_t nrows,
                        double *out) {
  if (N < 1 || D < 1 || !(scale > 0.0) || isinf(scale)) return -1;
  const double isd = scale;
  int64_t total = rows ? nrows : (int64_t)BH * N;
#pragma omp parallel
  {
    double *sc = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < total; r++) {
      int64_t id = rows ? rows[r] : r;
      int64_t bh = id / N;
      int i = (int)(id % N);
      const uint16_t *qi = q + ((size_t)bh * N + i) * D;
      int kend = causal ? i + 1 : N;
      double mx = -INFINITY;
      for (int j = 0; j < kend; j++) {
        const uint16_t *kj = k + ((size_t)bh * N + j) * D;
        double s = 0.0;
        for (int d = 0; d < D; d++) s += (double)bf16_to_f32(qi[d]) * (double)bf16_to_f32(kj[d]);
        sc[j] = s * isd;
        if (sc[j] > mx) mx = sc[j];
      }
      double sum = 0.0;
      for (int j = 0; j < kend; j++) {
        sc[j] = exp(sc[j] - mx);
        sum += sc[j];
      }
      double *o = out + (size_t)r * D;
      for (int d = 0; d < D; d++) o[d] = 0.0;
      for (int j = 0; j < kend; j++) {
        const uint16_t *vj = v + ((size_t)bh * N + j) * D;
        for (int d = 0; d < D; d++) o[d] += sc[j] * (double)bf16_to_f32(vj[d]);
      }
      for (int d = 0; d < D; d++) o[d] /= sum;
    }
    free(sc);
  }
  return 0;
}

int sor_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

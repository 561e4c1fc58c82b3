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

/* Q and K: groups of 16 consecutive elements along D, the contraction axis of
 * QK^T ([NEWS-OBST], solution 1).  No smoothing (mean subtraction) of K: the
 * pages do not describe one. */
void sor_quantize_rows(const uint16_t *x, int BH, int N, int D, uint8_t *codes, uint8_t *scales) {
  int N_pad = round_up(N, 128);
  size_t crow = (size_t)D / 2, srow = (size_t)D / 16;
  memset(codes, 0, (size_t)BH * N_pad * crow);
  memset(scales, 0, (size_t)BH * N_pad * srow);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < (int64_t)BH * N; r++) {
    int64_t bh = r / N, n = r % N;
    const uint16_t *src = x + (size_t)r * D;
    uint8_t *cdst = codes + ((size_t)bh * N_pad + n) * crow;
    uint8_t *sdst = scales + ((size_t)bh * N_pad + n) * srow;
    for (int g = 0; g < D / 16; g++) {
      float buf[16];
      uint8_t c[16];
      for (int i = 0; i < 16; i++) buf[i] = bf16_to_f32(src[g * 16 + i]);
      sor_quant_group16(buf, c, &sdst[g]);
      for (int i = 0; i < 16; i++) put_nibble(cdst, g * 16 + i, c[i]);
    }
  }
}

/* V: the contraction axis of PV is the token axis, so the 16-element groups
 * run along tokens for each channel (block scales of a block-scaled product
 * always run along the contraction axis).  Output is V^T.  Tokens past N are
 * zero, which makes an all-padding group's scale and codes zero. */
void sor_quantize_v(const uint16_t *v, int BH, int N, int D, uint8_t *codes, uint8_t *scales) {
  int N_pad = round_up(N, 128);
  size_t crow = (size_t)N_pad / 2, srow = (size_t)N_pad / 16;
  memset(codes, 0, (size_t)BH * D * crow);
  memset(scales, 0, (size_t)BH * D * srow);
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t bh = 0; bh < BH; bh++) {
    for (int d = 0; d < D; d++) {
      uint8_t *cdst = codes + ((size_t)bh * D + d) * crow;
      uint8_t *sdst = scales + ((size_t)bh * D + d) * srow;
      for (int g = 0; g < N_pad / 16; g++) {
        float buf[16];
        uint8_t c[16];
        for (int i = 0; i < 16; i++) {
          int n = g * 16 + i;
          buf[i] = (n < N) ? bf16_to_f32(v[((size_t)bh * N + n) * D + d]) : 0.0f;
        }
        sor_quant_group16(buf, c, &sdst[g]);
        for (int i = 0; i < 16; i++) put_nibble(cdst, g * 16 + i, c[i]);
      }
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Tiled attention with online softmax and two-level P quantization.         */
/* ------------------------------------------------------------------------ */

/* Decoding tables: the value of every E2M1 code and E4M3 byte, taken from the
 * codec definitions above. */
static double g_e2m1[16];
static double g_e4m3[256];
static int g_tables_ready = 0;

static void init_tables(void) {
  if (g_tables_ready) return;
#pragma omp critical(sor_tables)
  {
    if (!g_tables_ready) {
      for (int i = 0; i < 16; i++) g_e2m1[i] = sor_e2m1_value(i);
      for (int i = 0; i < 256; i++) g_e4m3[i] = sor_e4m3_value(i);
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
 *   level 2: the 1x16 group quantizer on P2 along keys (16 consecutive
 *            elements of a row, [NEWS-HW])
 *   acc    = acc * exp((m_old - m_new)/sqrt(D)) + sP1 * sum_j dec(P2_j) * dec(V_j)
 * and finally O = acc / l. */
static void attend_row(const uint8_t *qc, const uint8_t *qs, const uint8_t *kc, const uint8_t *ks,
                       const uint8_t *vc, const uint8_t *vs, int N, int N_pad, int D, int causal,
                       double scale, int pmode, int kv_tile, int i, double *out, double *out_l,
                       double *out_m) {
  const double isd = scale;
  const int G = D / 16;
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
        for (int k = 16 * g; k < 16 * g + 16; k++) part += qv[k] * g_e2m1[get_nibble(krow, k)];
        s += g_e4m3[qs[(size_t)i * G + g]] * g_e4m3[ks[(size_t)j * G + g]] * part;
      }
      S[jj] = s;
      if (s > t) t = s;
    }
    double m_new = (t > m) ? t : m;
    double alpha = exp((m - m_new) * isd);
    double lt = 0.0;
    for (int jj = 0; jj < T; jj++) lt += exp((S[jj] - m_new) * isd);
    l = l * alpha + lt;

    /* level 1 */
    double ref = (pmode == 0) ? t : m_new;
    double sP1 = (pmode == 0) ? exp((t - m_new) * isd) / 2688.0 : 1.0 / 2688.0;
    for (int jj = 0; jj < T; jj++) P2[jj] = (float)(2688.0 * exp((S[jj] - ref) * isd));
    /* level 2 */
    for (int g = 0; g < T / 16; g++) sor_quant_group16(&P2[16 * g], &pc[16 * g], &ps[g]);

    /* O update */
    for (int d = 0; d < D; d++) {
      const uint8_t *vrow = vc + (size_t)d * (N_pad / 2);
      const uint8_t *vsrow = vs + (size_t)d * (N_pad / 16);
      double pv = 0.0;
      for (int g = 0; g < T / 16; g++) {
        int jg = (j0 / 16) + g; /* token group index */
        if (16 * jg >= N_pad) break;
        double part = 0.0;
        for (int k = 0; k < 16; k++)
          part += g_e2m1[pc[16 * g + k]] * g_e2m1[get_nibble(vrow, 16 * jg + k)];
        pv += g_e4m3[ps[g]] * g_e4m3[vsrow[jg]] * part;
      }
      acc[d] = acc[d] * alpha + sP1 * pv;
    }
    m = m_new;
  }
  for (int d = 0; d < D; d++) out[d] = acc[d] / l;
  if (out_l) *out_l = l;
  if (out_m) *out_m = m;
}

int sor_attention(const uint8_t *qc, const uint8_t *qs, const uint8_t *kc, const uint8_t *ks,
                  const uint8_t *vc, const uint8_t *vs, int BH, int N, int D, int causal,
                  double scale, int pmode, int kv_tile, const int64_t *rows, int64_t nrows,
                  double *out, double *out_l, double *out_m) {
  if (D % 16 || D > SOR_MAX_D || kv_tile % 16 || kv_tile > SOR_MAX_TILE || kv_tile <= 0 || N < 1 ||
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
    attend_row(qc + (size_t)bh * N_pad * (D / 2), qs + (size_t)bh * N_pad * (D / 16),
               kc + (size_t)bh * N_pad * (D / 2), ks + (size_t)bh * N_pad * (D / 16),
               vc + (size_t)bh * D * (N_pad / 2), vs + (size_t)bh * D * (N_pad / 16), N, N_pad, D,
               causal, scale, pmode, kv_tile, i, out + (size_t)r * D, out_l ? out_l + r : 0,
               out_m ? out_m + r : 0);
  }
  return 0;
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

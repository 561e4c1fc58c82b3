/*
 * sagebwd_oracle.c -- CPU oracle for SageBwd, the 8-bit attention for
 * training (senqingzn.com article on SageAttention3, "INT8 attention for
 * training" and "Solving two obstacles and one difficulty", difficulty 3).
 * TEST INFRASTRUCTURE ONLY (tests and the bench's CPU baseline).
 *
 * The pages fix three things: six of the seven matrix products of attention
 * training run in INT8; of the five products of the backward pass, the one
 * most sensitive to precision is kept at FP16; the attention-map gradient is
 * the quantity whose quantization error accumulates.  Everything else is a
 * reading, stated where it is used:
 *
 *   products  forward  S = Q K^T, O = P V;  backward  S = Q K^T (recomputed),
 *             dV = P^T dO, dP = dO V^T, dQ = dS K, dK = dS^T Q.  dP = dO V^T,
 *             the product that gives the attention-map gradient, is the FP16
 *             one (inputs rounded to FP16, exact products, summed in double
 *             here); the other six are INT8.
 *   INT8      symmetric, per block: s = amax / 127 (float division), codes
 *             rint(x * (127 / amax)) (float division and product, rounded to
 *             nearest even), clamped to [-127, 127]; an all-zero block has
 *             s = 0 and codes 0.  Q, K, V and dO: per head, blocks of 128
 *             tokens over all D channels.  P and dS: blocks of 64 queries x
 *             128 keys (aligned to multiples of 64 and 128; the last ones
 *             ragged), so that each block's scale is constant along both
 *             contractions it enters.
 *   forward   FlashAttention's online softmax over key tiles of 128, in key
 *             order.  For each row, m is the running maximum of scale * S
 *             including the current tile; the tile's probabilities
 *             P~ = exp(scale * S - m) (masked entries 0, rounded to float) are
 *             INT8-quantized per block and enter O through the INT8 product;
 *             the normaliser l sums the unquantized P~.  O and l are rescaled
 *             by exp(m_old - m_new) when m grows.  The forward saves
 *             L = m + log(l) and returns O / l.
 *   backward  P = exp(scale * S - L) exactly (masked 0), from the same
 *             quantized Q and K; D_i = sum_d dO_id O_id with the O the forward
 *             returns (rounded to bf16); dS = P o (dP - D);
 *             dV = P^^T dO^, dQ = scale * dS^ K^, dK = scale * dS^^T Q^, the
 *             hats being the INT8 blocks above.
 *   causal    key j is visible from query i when j <= i.
 *
 * quant = 0 skips every rounding step (INT8, FP16, bf16, float): the result
 * is then float64 softmax attention and its exact gradient, which pins the
 * algebra.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off (no fast-math), like the
 * SageAttention3 oracle in sage_oracle.c, with which it shares no code.
 */
#include "sagebwd_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define TOK 128 /* token block of Q, K, V, dO; key edge of a P / dS block */
#define QBLK 64 /* query edge of a P / dS block */

static float bf16f(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a double to the nearest bf16 value (ties to even), as a double. */
static double bf16_round(double x) {
  if (x == 0.0 || isnan(x) || isinf(x)) return x;
  int e;
  frexp(x, &e); /* |x| = f * 2^e, f in [0.5, 1): 8 significant bits */
  double ulp = ldexp(1.0, e - 8);
  return rint(x / ulp) * ulp;
}

/* Round a float to the nearest FP16 value (ties to even), as a double.
 * Magnitudes past the largest finite FP16 value saturate to it. */
static double fp16_round(float x) {
  if (x == 0.0f || isnan(x)) return (double)x;
  double a = fabs((double)x), r;
  if (a >= 65504.0) {
    r = 65504.0;
  } else if (a < ldexp(1.0, -14)) {
    r = rint(a * ldexp(1.0, 24)) * ldexp(1.0, -24); /* subnormal step 2^-24 */
  } else {
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): 11 significant bits */
    double ulp = ldexp(1.0, e - 11);
    r = rint(a / ulp) * ulp;
  }
  return x < 0 ? -r : r;
}

/* INT8 code of x in a block of absolute maximum amax (the reading above). */
int sbo_int8_code(float x, float amax) {
  if (amax == 0.0f) return 0;
  float inv = 127.0f / amax;
  float y = x * inv;
  float c = rintf(y);
  if (c > 127.0f) c = 127.0f;
  if (c < -127.0f) c = -127.0f;
  return (int)c;
}

float sbo_int8_scale(float amax) { return amax / 127.0f; }

/* bf16 [BH][N][D] -> codes [BH][N][D], one scale per (head, 128-token block). */
void sbo_quantize_blocks(const uint16_t *x, int BH, int N, int D, int8_t *codes, float *scales) {
  const int nb = (N + TOK - 1) / TOK;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t bh = 0; bh < BH; bh++)
    for (int b = 0; b < nb; b++) {
      const int n0 = b * TOK, n1 = (n0 + TOK < N) ? n0 + TOK : N;
      float amax = 0.0f;
      for (int n = n0; n < n1; n++)
        for (int d = 0; d < D; d++) {
          float a = fabsf(bf16f(x[((size_t)bh * N + n) * D + d]));
          if (a > amax) amax = a;
        }
      scales[(size_t)bh * nb + b] = sbo_int8_scale(amax);
      for (int n = n0; n < n1; n++)
        for (int d = 0; d < D; d++) {
          size_t i = ((size_t)bh * N + n) * D + d;
          codes[i] = (int8_t)sbo_int8_code(bf16f(x[i]), amax);
        }
    }
}

/* Dequantized values of a bf16 tensor's head: INT8 per 128-token block, or the
 * bf16 values themselves when quant = 0. */
static void dequant_head(const uint16_t *x, int N, int D, int quant, double *out) {
  const int nb = (N + TOK - 1) / TOK;
  for (int b = 0; b < nb; b++) {
    const int n0 = b * TOK, n1 = (n0 + TOK < N) ? n0 + TOK : N;
    float amax = 0.0f;
    for (int n = n0; n < n1; n++)
      for (int d = 0; d < D; d++) {
        float a = fabsf(bf16f(x[(size_t)n * D + d]));
        if (a > amax) amax = a;
      }
    const double s = (double)sbo_int8_scale(amax);
    for (int n = n0; n < n1; n++)
      for (int d = 0; d < D; d++) {
        float v = bf16f(x[(size_t)n * D + d]);
        out[(size_t)n * D + d] = quant ? s * sbo_int8_code(v, amax) : (double)v;
      }
  }
}

/* Quantize rows [i0, i1) x columns [j0, j1) of the [N][N] matrix m as one
 * INT8 block (values rounded to float first); out = dequantized values. */
static void quant_block(const double *m, int N, int i0, int i1, int j0, int j1, int quant, double *out) {
  if (!quant) {
    for (int i = i0; i < i1; i++)
      for (int j = j0; j < j1; j++) out[(size_t)i * N + j] = m[(size_t)i * N + j];
    return;
  }
  float amax = 0.0f;
  for (int i = i0; i < i1; i++)
    for (int j = j0; j < j1; j++) {
      float a = fabsf((float)m[(size_t)i * N + j]);
      if (a > amax) amax = a;
    }
  const double s = (double)sbo_int8_scale(amax);
  for (int i = i0; i < i1; i++)
    for (int j = j0; j < j1; j++) out[(size_t)i * N + j] = s * sbo_int8_code((float)m[(size_t)i * N + j], amax);
}

/* The whole [N][N] matrix, block by block (64 queries x 128 keys). */
static void quant_blocks_nn(const double *m, int N, int quant, double *out) {
#pragma omp parallel for schedule(static)
  for (int i0 = 0; i0 < N; i0 += QBLK)
    for (int j0 = 0; j0 < N; j0 += TOK)
      quant_block(m, N, i0, (i0 + QBLK < N) ? i0 + QBLK : N, j0, (j0 + TOK < N) ? j0 + TOK : N, quant, out);
}

/* dst[j][d] = sum over i (ascending) of M[i][j] * X[i][d], for the [N][N]
 * matrix M and [N][D] X: the transposed products dV and dK.  Threads take
 * disjoint ranges of j; each sum keeps its order. */
static void mt_times(const double *M, const double *X, int N, int D, double *dst) {
#pragma omp parallel for schedule(static)
  for (int jb = 0; jb < N; jb += 32) {
    const int je = (jb + 32 < N) ? jb + 32 : N;
    for (int j = jb; j < je; j++)
      for (int d = 0; d < D; d++) dst[(size_t)j * D + d] = 0.0;
    for (int i = 0; i < N; i++)
      for (int j = jb; j < je; j++)
        for (int d = 0; d < D; d++) dst[(size_t)j * D + d] += M[(size_t)i * N + j] * X[(size_t)i * D + d];
  }
}

/* One head.  The heads run one after another; the loops inside run their
 * independent rows (or row blocks) in parallel, every sum in a fixed order. */
static int train_head(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout, int N, int D,
                      int causal, double scale, int quant, double *O, double *lse, double *dq, double *dk,
                      double *dv) {
  double *Qd = malloc(sizeof(double) * N * D), *Kd = malloc(sizeof(double) * N * D);
  double *Vd = malloc(sizeof(double) * N * D), *dOd = malloc(sizeof(double) * N * D);
  double *S = malloc(sizeof(double) * N * N), *P = malloc(sizeof(double) * N * N);
  double *Pq = malloc(sizeof(double) * N * N), *L = malloc(sizeof(double) * N);
  double *Dr = malloc(sizeof(double) * N), *m = malloc(sizeof(double) * N);
  double *l = malloc(sizeof(double) * N);
  double *dOh = malloc(sizeof(double) * N * D), *Vh = malloc(sizeof(double) * N * D);
  int rc = 0;
  if (!Qd || !Kd || !Vd || !dOd || !S || !P || !Pq || !L || !Dr || !m || !l || !dOh || !Vh) {
    rc = -2;
    goto out;
  }
  dequant_head(q, N, D, quant, Qd);
  dequant_head(k, N, D, quant, Kd);
  dequant_head(v, N, D, quant, Vd);
  dequant_head(dout, N, D, quant, dOd);
  /* scale * S = scale * Q^ K^^T (an INT8 product; exact here), masked -inf */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < N; i++)
    for (int j = 0; j < N; j++) {
      double s = 0.0;
      for (int d = 0; d < D; d++) s += Qd[(size_t)i * D + d] * Kd[(size_t)j * D + d];
      S[(size_t)i * N + j] = (causal && j > i) ? -INFINITY : scale * s;
    }
  /* forward: online softmax over key tiles; P~ of each tile into P */
  for (size_t x = 0; x < (size_t)N * D; x++) O[x] = 0.0;
  for (int i = 0; i < N; i++) {
    m[i] = -INFINITY;
    l[i] = 0.0;
  }
  for (int j0 = 0; j0 < N; j0 += TOK) {
    const int j1 = (j0 + TOK < N) ? j0 + TOK : N;
#pragma omp parallel for schedule(static)
    for (int i = 0; i < N; i++) {
      double mt = -INFINITY;
      for (int j = j0; j < j1; j++)
        if (S[(size_t)i * N + j] > mt) mt = S[(size_t)i * N + j];
      const double mn = (mt > m[i]) ? mt : m[i];
      const double alpha = (m[i] == -INFINITY) ? 0.0 : exp(m[i] - mn);
      double rs = 0.0;
      for (int j = j0; j < j1; j++) {
        double s = S[(size_t)i * N + j];
        double p = (s == -INFINITY) ? 0.0 : exp(s - mn);
        if (quant) p = (double)(float)p;
        P[(size_t)i * N + j] = p;
        rs += p;
      }
      l[i] = l[i] * alpha + rs;
      for (int d = 0; d < D; d++) O[(size_t)i * D + d] *= alpha;
      m[i] = mn;
    }
    /* O += P~^ V^ for this key tile, P~ quantized per (64 x 128) block; each
     * sum runs over j in ascending order */
#pragma omp parallel for schedule(static)
    for (int i0 = 0; i0 < N; i0 += QBLK) {
      const int i1 = (i0 + QBLK < N) ? i0 + QBLK : N;
      double acc[D];
      quant_block(P, N, i0, i1, j0, j1, quant, Pq);
      for (int i = i0; i < i1; i++) {
        for (int d = 0; d < D; d++) acc[d] = 0.0;
        for (int j = j0; j < j1; j++)
          for (int d = 0; d < D; d++) acc[d] += Pq[(size_t)i * N + j] * Vd[(size_t)j * D + d];
        for (int d = 0; d < D; d++) O[(size_t)i * D + d] += acc[d];
      }
    }
  }
  for (int i = 0; i < N; i++) {
    L[i] = m[i] + log(l[i]);
    lse[i] = L[i];
    for (int d = 0; d < D; d++) O[(size_t)i * D + d] /= l[i];
  }
  /* backward: exact P from L (the forward's quantized Q and K) */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < N; i++)
    for (int j = 0; j < N; j++) {
      double s = S[(size_t)i * N + j];
      P[(size_t)i * N + j] = (s == -INFINITY) ? 0.0 : exp(s - L[i]);
    }
  /* dV = P^^T dO^ (INT8) */
  quant_blocks_nn(P, N, quant, Pq);
  mt_times(Pq, dOd, N, D, dv);
  /* D_i = rowsum(dO o O), O as the forward returns it */
  for (int i = 0; i < N; i++) {
    double r = 0.0;
    for (int d = 0; d < D; d++) {
      double od = O[(size_t)i * D + d];
      r += (double)bf16f(dout[(size_t)i * D + d]) * (quant ? bf16_round(od) : od);
    }
    Dr[i] = r;
  }
  /* dP = dO V^T in FP16 (inputs rounded to FP16); dS = P o (dP - D) into S */
  for (size_t x = 0; x < (size_t)N * D; x++) {
    float a = bf16f(dout[x]), b = bf16f(v[x]);
    dOh[x] = quant ? fp16_round(a) : (double)a;
    Vh[x] = quant ? fp16_round(b) : (double)b;
  }
#pragma omp parallel for schedule(static)
  for (int i = 0; i < N; i++)
    for (int j = 0; j < N; j++) {
      double dp = 0.0;
      for (int d = 0; d < D; d++) dp += dOh[(size_t)i * D + d] * Vh[(size_t)j * D + d];
      S[(size_t)i * N + j] = P[(size_t)i * N + j] * (dp - Dr[i]);
    }
  /* dQ = scale * dS^ K^, dK = scale * dS^^T Q^ (INT8) */
  quant_blocks_nn(S, N, quant, Pq);
#pragma omp parallel for schedule(static)
  for (int i = 0; i < N; i++) {
    double acc[D];
    for (int d = 0; d < D; d++) acc[d] = 0.0;
    for (int j = 0; j < N; j++)
      for (int d = 0; d < D; d++) acc[d] += Pq[(size_t)i * N + j] * Kd[(size_t)j * D + d];
    for (int d = 0; d < D; d++) dq[(size_t)i * D + d] = scale * acc[d];
  }
  mt_times(Pq, Qd, N, D, dk);
  for (size_t x = 0; x < (size_t)N * D; x++) dk[x] *= scale;
out:
  free(Qd);
  free(Kd);
  free(Vd);
  free(dOd);
  free(S);
  free(P);
  free(Pq);
  free(L);
  free(Dr);
  free(m);
  free(l);
  free(dOh);
  free(Vh);
  return rc;
}

int sbo_attention_train(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                        int BH, int N, int D, int causal, double scale, int quant, double *o,
                        double *lse, double *dq, double *dk, double *dv) {
  if (BH < 0 || N < 1 || D < 1 || D > 4096 || !(scale > 0.0) || isinf(scale) || (quant != 0 && quant != 1))
    return -1;
  for (int64_t bh = 0; bh < BH; bh++) {
    const size_t hoff = (size_t)bh * N * D;
    int rc = train_head(q + hoff, k + hoff, v + hoff, dout + hoff, N, D, causal, scale, quant, o + hoff,
                        lse + (size_t)bh * N, dq + hoff, dk + hoff, dv + hoff);
    if (rc) return rc;
  }
  return 0;
}

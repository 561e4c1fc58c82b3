/* oracle_driver.c -- drives every entry point of the CPU oracle over small,
 * ragged shapes so that a build with -fsanitize=address,undefined can check
 * its memory accesses and arithmetic (tests/test_sanitizers.py).  Test
 * infrastructure: it checks return codes and that outputs are finite, not
 * values (the pins in tests/test_oracle_*.py do that). */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "sage_oracle.h"
#include "sagebwd_oracle.h"

static unsigned long long rng_state = 0x9E3779B97F4A7C15ull;

static unsigned rnd(void) {
  rng_state ^= rng_state << 13;
  rng_state ^= rng_state >> 7;
  rng_state ^= rng_state << 17;
  return (unsigned)(rng_state >> 16);
}

/* a bf16 bit pattern of a value of magnitude up to about 2^e */
static unsigned short bf16_rand(int e) {
  float x = ldexpf((float)((int)(rnd() % 2001) - 1000) / 1000.0f, (int)(rnd() % (unsigned)(e + 1)));
  unsigned u;
  memcpy(&u, &x, 4);
  return (unsigned short)(u >> 16);
}

static int fail(const char *what) {
  fprintf(stderr, "oracle driver: %s\n", what);
  return 1;
}

static int run_shape(int BH, int N, int D, int fmt) {
  const int Np = (N + 127) / 128 * 128;
  const int G = fmt ? 32 : 16;
  const size_t elems = (size_t)BH * N * D;
  unsigned short *q = malloc(elems * 2), *k = malloc(elems * 2), *v = malloc(elems * 2);
  uint8_t *qc = malloc((size_t)BH * Np * D / 2), *qs = malloc((size_t)BH * Np * D / G);
  uint8_t *kc = malloc((size_t)BH * Np * D / 2), *ks = malloc((size_t)BH * Np * D / G);
  uint8_t *vc = malloc((size_t)BH * D * Np / 2), *vs = malloc((size_t)BH * D * Np / G);
  /* room for every row, or for the row subset below (up to 64 rows, repeats allowed) */
  const size_t nout = (size_t)BH * N > 64 ? (size_t)BH * N : 64;
  double *out = malloc(nout * D * sizeof(double)), *ol = malloc(nout * sizeof(double));
  double *om = malloc(nout * sizeof(double));
  for (size_t i = 0; i < elems; i++) {
    q[i] = bf16_rand(2);
    k[i] = bf16_rand(4);
    v[i] = bf16_rand(1);
  }
  sor_quantize_rows_fmt(q, BH, N, D, fmt, qc, qs);
  sor_quantize_rows_fmt(k, BH, N, D, fmt, kc, ks);
  sor_quantize_v_fmt(v, BH, N, D, fmt, vc, vs);
  if (!fmt) {
    /* the NVFP4-only entry points are the same quantizers */
    sor_quantize_rows(q, BH, N, D, qc, qs);
    sor_quantize_v(v, BH, N, D, vc, vs);
  }
  const double scale = 1.0 / sqrt((double)D);
  for (int causal = 0; causal < 2; causal++)
    for (int pmode = 0; pmode < 2; pmode++)
      for (int lnorm = 0; lnorm < 2; lnorm++) {
        if (sor_attention_ex(qc, qs, kc, ks, vc, vs, BH, N, D, causal, fmt, scale, pmode, lnorm, 128,
                             NULL, 0, out, ol, om) != 0)
          return fail("attention rejected valid arguments");
        for (size_t i = 0; i < elems; i++)
          if (!isfinite(out[i])) return fail("non-finite attention output");
      }
  /* a row subset, the first and the last row of every head */
  int64_t rows[64];
  int64_t nrows = 0;
  for (int b = 0; b < BH && nrows < 62; b++) {
    rows[nrows++] = (int64_t)b * N;
    rows[nrows++] = (int64_t)b * N + N - 1;
  }
  if (sor_attention(qc, qs, kc, ks, vc, vs, BH, N, D, 1, fmt, scale, 0, 128, rows, nrows, out, ol, om) != 0)
    return fail("attention rejected a row subset");
  if (sor_attention_exact(q, k, v, BH, N, D, 1, scale, rows, nrows, out) != 0)
    return fail("exact attention rejected valid arguments");
  if (sor_attention_exact(q, k, v, BH, N, D, 0, scale, NULL, 0, out) != 0)
    return fail("exact attention rejected valid arguments");
  /* rejected arguments */
  if (sor_attention_ex(qc, qs, kc, ks, vc, vs, BH, N, D, 0, 2, scale, 0, 0, 128, NULL, 0, out, ol, om) != -1 ||
      sor_attention_ex(qc, qs, kc, ks, vc, vs, BH, N, D, 0, fmt, scale, 0, 2, 128, NULL, 0, out, ol, om) != -1 ||
      sor_attention_ex(qc, qs, kc, ks, vc, vs, BH, N, D, 0, fmt, scale, 0, 0, 1024, NULL, 0, out, ol, om) != -1 ||
      sor_attention_ex(qc, qs, kc, ks, vc, vs, BH, N, D, 0, fmt, -1.0, 0, 0, 128, NULL, 0, out, ol, om) != -1 ||
      sor_attention_exact(q, k, v, BH, N, D, 0, 0.0, NULL, 0, out) != -1)
    return fail("an invalid argument was accepted");
  free(q);
  free(k);
  free(v);
  free(qc);
  free(qs);
  free(kc);
  free(ks);
  free(vc);
  free(vs);
  free(out);
  free(ol);
  free(om);
  return 0;
}

/* SageBwd forward and backward, both modes, causal and not */
static int run_train(int BH, int N, int D) {
  const size_t elems = (size_t)BH * N * D;
  unsigned short *x[4];
  for (int t = 0; t < 4; t++) {
    x[t] = malloc(elems * 2);
    for (size_t i = 0; i < elems; i++) x[t][i] = bf16_rand(3);
  }
  double *out[5];
  for (int t = 0; t < 5; t++) out[t] = malloc(sizeof(double) * (t == 1 ? (size_t)BH * N : elems));
  int8_t *codes = malloc(elems);
  float *scales = malloc(sizeof(float) * BH * ((N + 127) / 128));
  sbo_quantize_blocks(x[0], BH, N, D, codes, scales);
  for (int quant = 0; quant < 2; quant++)
    for (int causal = 0; causal < 2; causal++) {
      if (sbo_attention_train(x[0], x[1], x[2], x[3], BH, N, D, causal, 0.125, quant, out[0], out[1], out[2],
                              out[3], out[4]))
        return fail("SageBwd oracle rejected valid arguments");
      for (int t = 0; t < 5; t++)
        for (size_t i = 0; i < (t == 1 ? (size_t)BH * N : elems); i++)
          if (!isfinite(out[t][i])) return fail("non-finite SageBwd output");
    }
  if (sbo_attention_train(x[0], x[1], x[2], x[3], BH, 0, D, 0, 0.125, 1, out[0], out[1], out[2], out[3],
                          out[4]) != -1)
    return fail("SageBwd oracle accepted N = 0");
  for (int t = 0; t < 4; t++) free(x[t]);
  for (int t = 0; t < 5; t++) free(out[t]);
  free(codes);
  free(scales);
  return 0;
}

int main(void) {
  /* codecs over a range of float32 patterns, and every E4M3 / E8M0 byte */
  enum { R = 1 << 16 };
  uint8_t *e2 = malloc(R), *e4 = malloc(R);
  const unsigned firsts[] = {0u, 0x3E000000u, 0x3F800000u, 0x43E00000u, 0x7F7F0000u, 0x80000000u, 0xBF000000u};
  for (unsigned i = 0; i < sizeof firsts / sizeof firsts[0]; i++) sor_encode_range(firsts[i], R, e2, e4);
  for (int b = 0; b < 256; b++) {
    (void)sor_e4m3_value(b);
    (void)sor_e8m0_value(b);
  }
  for (int c = 0; c < 16; c++) (void)sor_e2m1_value(c);
  /* the group quantizers on random groups, zeros and extremes */
  for (int t = 0; t < 2000; t++) {
    float x[32];
    uint8_t codes[32], sc;
    for (int i = 0; i < 32; i++) x[i] = ldexpf((float)((int)(rnd() % 2001) - 1000), (int)(rnd() % 60) - 40);
    if (t % 7 == 0) memset(x, 0, sizeof x);
    sor_quant_group16(x, codes, &sc);
    sor_quant_group32_mx(x, codes, &sc);
  }
  free(e2);
  free(e4);
  const int shapes[][3] = {{1, 1, 64}, {2, 17, 64}, {1, 130, 128}, {2, 257, 64}, {1, 300, 128}};
  for (unsigned s = 0; s < sizeof shapes / sizeof shapes[0]; s++)
    for (int fmt = 0; fmt < 2; fmt++)
      if (run_shape(shapes[s][0], shapes[s][1], shapes[s][2], fmt)) return 1;
  const int train_shapes[][3] = {{1, 1, 64}, {2, 65, 64}, {1, 200, 128}};
  for (unsigned s = 0; s < sizeof train_shapes / sizeof train_shapes[0]; s++)
    if (run_train(train_shapes[s][0], train_shapes[s][1], train_shapes[s][2])) return 1;
  printf("oracle driver: ok\n");
  return 0;
}

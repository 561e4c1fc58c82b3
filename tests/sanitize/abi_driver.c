/* abi_driver.c -- drives the C ABI of include/sage_fp4.h through every path
 * that returns before any device work: argument rejections, size overflows,
 * empty problems, workspace carving and the status strings.  Built with
 * -fsanitize=address,undefined against a library whose host code is built the
 * same way (tests/test_sanitizers.py), so that the argument checks' own
 * arithmetic and memory accesses are checked.  No GPU is needed: pointers
 * passed here are aligned placeholders that the rejected calls never touch. */
#include <limits.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "sage_fp4.h"
#include "sagebwd.h"

static int failures = 0;

static void expect(int got, int want, const char *what) {
  if (got != want) {
    fprintf(stderr, "abi driver: %s: got %d, want %d\n", what, got, want);
    failures++;
  }
}

#define P(x) ((void *)(uintptr_t)(x))

int main(void) {
  /* workspace sizes: valid, invalid and overflowing shapes */
  if (sage_fp4_workspace_bytes(4, 32, 4096, 128) == 0) expect(0, 1, "workspace of the LLM shape");
  expect((int)sage_fp4_workspace_bytes(1, 1, 17, 96), 0, "workspace, D = 96");
  expect((int)sage_fp4_workspace_bytes(-1, 1, 17, 64), 0, "workspace, B < 0");
  expect((int)sage_fp4_workspace_bytes(INT_MAX, INT_MAX, INT_MAX, 128), 0, "workspace, overflowing sizes");
  expect((int)sage_fp4_workspace_bytes(65536, 65536, 4096, 64), 0, "workspace, B*H*N past 32 bits");
  expect((int)sage_fp4_host_workspace_bytes(INT_MAX, INT_MAX, 4096, 64), 0, "host workspace, overflow");
  expect((int)sage_fp4_host_workspace_bytes(1, 1, 17, 80), 0, "host workspace, D = 80");

  /* carving a real host buffer (pointer arithmetic only) */
  const int B = 2, H = 3, N = 300, D = 64;
  const size_t ws = sage_fp4_workspace_bytes(B, H, N, D);
  uint8_t *buf = aligned_alloc(256, (ws + 255) / 256 * 256);
  sage_fp4_qkv qkv;
  expect(sage_fp4_qkv_from_workspace(buf, ws, B, H, N, D, &qkv), SAGE_FP4_OK, "carve workspace");
  expect(sage_fp4_qkv_from_workspace(buf, ws - 1, B, H, N, D, &qkv), SAGE_FP4_EINVAL, "carve, short");
  expect(sage_fp4_qkv_from_workspace(buf + 16, ws, B, H, N, D, &qkv), SAGE_FP4_EINVAL, "carve, misaligned");
  expect(sage_fp4_qkv_from_workspace(buf, ws, B, H, N, D, NULL), SAGE_FP4_EINVAL, "carve, no output");
  expect(sage_fp4_qkv_from_workspace(buf, ws, B, H, N, D, &qkv), SAGE_FP4_OK, "carve again");

  /* quantize: bad pointers, shapes, formats, strides; empty problems */
  expect(sage_fp4_quantize_qkv(NULL, P(0x2000), P(0x3000), &qkv, B, H, N, D, NULL), SAGE_FP4_EINVAL, "quant q null");
  expect(sage_fp4_quantize_qkv(P(0x1004), P(0x2000), P(0x3000), &qkv, B, H, N, D, NULL), SAGE_FP4_EINVAL,
         "quant q misaligned");
  expect(sage_fp4_quantize_qkv(P(0x1000), P(0x2000), P(0x3000), NULL, B, H, N, D, NULL), SAGE_FP4_EINVAL,
         "quant no operands");
  expect(sage_fp4_quantize_qkv(P(0x1000), P(0x2000), P(0x3000), &qkv, B, H, N, 80, NULL), SAGE_FP4_EINVAL,
         "quant D = 80");
  expect(sage_fp4_quantize_qkv(P(0x1000), P(0x2000), P(0x3000), &qkv, 0, H, N, D, NULL), SAGE_FP4_OK,
         "quant empty batch");
  expect(sage_fp4_quantize_qkv(P(0x1000), P(0x2000), P(0x3000), &qkv, B, H, 0, D, NULL), SAGE_FP4_OK,
         "quant empty sequence");
  sage_fp4_strides bad = {8, 8, 12};
  sage_fp4_strides huge = {INT64_MAX / 2 + 8, 8, 8};
  sage_fp4_strides neg = {-8, 8, 8};
  expect(sage_fp4_quantize_qkv_strided(P(0x1000), &bad, P(0x2000), NULL, P(0x3000), NULL, &qkv, B, H, N, D,
                                       SAGE_FP4_FORMAT_NVFP4, NULL),
         SAGE_FP4_EINVAL, "quant stride not a multiple of 8");
  expect(sage_fp4_quantize_qkv_strided(P(0x1000), &huge, P(0x2000), NULL, P(0x3000), NULL, &qkv, B, H, N, D,
                                       SAGE_FP4_FORMAT_NVFP4, NULL),
         SAGE_FP4_EINVAL, "quant stride overflow");
  expect(sage_fp4_quantize_qkv_strided(P(0x1000), NULL, P(0x2000), &neg, P(0x3000), NULL, &qkv, B, H, N, D,
                                       SAGE_FP4_FORMAT_NVFP4, NULL),
         SAGE_FP4_EINVAL, "quant negative stride");
  expect(sage_fp4_quantize_qkv_strided(P(0x1000), NULL, P(0x2000), NULL, P(0x3000), NULL, &qkv, B, H, N, D, 7,
                                       NULL),
         SAGE_FP4_EINVAL, "quant unknown format");
  expect(sage_fp4_quantize_qkv_stall_test(P(0x1000), P(0x2000), P(0x3000), &qkv, B, H, N, D, 10, NULL),
         SAGE_FP4_EINVAL, "quant stall limit too short");

  /* attention */
  expect(sage_fp4_attn_fwd(&qkv, NULL, B, H, N, D, 0, NULL), SAGE_FP4_EINVAL, "attn o null");
  expect(sage_fp4_attn_fwd(&qkv, P(0x4008), B, H, N, D, 0, NULL), SAGE_FP4_EINVAL, "attn o misaligned");
  expect(sage_fp4_attn_fwd(&qkv, P(0x4000), B, H, N, D, 2, NULL), SAGE_FP4_EINVAL, "attn causal = 2");
  expect(sage_fp4_attn_fwd(NULL, P(0x4000), B, H, N, D, 0, NULL), SAGE_FP4_EINVAL, "attn no operands");
  expect(sage_fp4_attn_fwd(&qkv, P(0x4000), 0, H, N, D, 0, NULL), SAGE_FP4_OK, "attn empty");
  expect(sage_fp4_attn_fwd_ex(&qkv, P(0x4000), NULL, B, H, N, D, 0, 0.0f, 0, NULL), SAGE_FP4_EINVAL,
         "attn scale 0");
  expect(sage_fp4_attn_fwd_ex(&qkv, P(0x4000), NULL, B, H, N, D, 0, 2e30f, 0, NULL), SAGE_FP4_EINVAL,
         "attn scale too large");
  expect(sage_fp4_attn_fwd_ex(&qkv, P(0x4000), &bad, B, H, N, D, 0, 0.1f, 0, NULL), SAGE_FP4_EINVAL,
         "attn O stride");
  sage_fp4_strides nhd = {(int64_t)N * H * D, D, (int64_t)H * D};
  expect(sage_fp4_attn_fwd_ex(&qkv, P(0x4000), &nhd, B, H, N, D, 0, 0.1f, SAGE_FP4_FORMAT_MXFP4_DIRECTP, NULL),
         SAGE_FP4_EINVAL, "attn Direct-P with strided O");
  expect(sage_fp4_attn_fwd_stall_test(&qkv, P(0x4000), B, H, N, D, 0, 1, NULL), SAGE_FP4_EINVAL,
         "attn stall limit too short");
  sage_fp4_qkv broken = qkv;
  broken.vt.scales = (uint8_t *)broken.vt.scales + 8;
  expect(sage_fp4_attn_fwd(&broken, P(0x4000), B, H, N, D, 0, NULL), SAGE_FP4_EINVAL, "attn misaligned scales");
  expect(sage_fp4_get_status(NULL, NULL), SAGE_FP4_EINVAL, "status, no operands");

  /* the one-call paths */
  expect(sage_fp4_attention_noalloc(P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5000), 4, 32, 4096, 128, 0,
                                    NULL),
         SAGE_FP4_ETOOLARGE, "noalloc too large");
  expect(sage_fp4_attention_noalloc(P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5002), 1, 2, 512, 128, 0,
                                    NULL),
         SAGE_FP4_EINVAL, "noalloc status misaligned");
  expect(sage_fp4_attention_noalloc(P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5000), 0, 2, 512, 128, 0,
                                    NULL),
         SAGE_FP4_OK, "noalloc empty");
  expect(sage_fp4_attention_host(P(0x1000), P(0x2000), P(0x3000), P(0x4000), B, H, N, D, 0, P(0x100000), 16,
                                 P(0x5000), NULL),
         SAGE_FP4_EINVAL, "host path, workspace too small");
  expect(sage_fp4_attention_host(P(0x1000), P(0x2000), P(0x3000), P(0x4000), 0, H, N, D, 0, P(0x100000), 256,
                                 P(0x5000), NULL),
         SAGE_FP4_OK, "host path, empty");

  /* diagnostics: rejected shapes and flags */
  expect(sage_fp4_cvt_probe(0, 16, NULL, NULL, NULL), SAGE_FP4_EINVAL, "cvt probe, no outputs");
  expect(sage_fp4_cvt_probe(0, 0, P(0x1000), NULL, NULL), SAGE_FP4_OK, "cvt probe, nothing to do");
  expect(sage_fp4_mma_probe(P(0x1000), P(0x2000), P(0x3000), P(0x4000), 96, 64, 0, P(0x5000), P(0x6000), NULL),
         SAGE_FP4_EINVAL, "mma probe n = 96");
  expect(sage_fp4_mma_probe_ex(P(0x1000), P(0x2000), P(0x3000), P(0x4000), 128, 64, 8, P(0x5000), P(0x6000),
                               NULL),
         SAGE_FP4_EINVAL, "mma probe unknown flag");
  expect(sage_fp4_mma_peak(0, 128, P(0x5000), NULL), SAGE_FP4_EINVAL, "mma peak, no iterations");
  expect(sage_fp4_tmem_max_probe(NULL, P(0x2000), P(0x3000), NULL), SAGE_FP4_EINVAL, "tmem probe, no input");

  /* SageBwd (include/sagebwd.h): workspace layout and argument rejections */
  {
    size_t offs[SAGEBWD_WS_FIELDS];
    const size_t sb = sagebwd_workspace_bytes(2, 3, 300, 64);
    if (sb == 0 || sagebwd_workspace_layout(2, 3, 300, 64, offs) != SAGE_FP4_OK) expect(0, 1, "sagebwd layout");
    for (int i = 1; i < SAGEBWD_WS_FIELDS; i++)
      if (offs[i] <= offs[i - 1] || offs[i] % 256 || offs[i] >= sb) expect(i, -1, "sagebwd offsets increase");
    expect((int)sagebwd_workspace_bytes(INT_MAX, INT_MAX, INT_MAX, 128), 0, "sagebwd workspace, overflow");
    expect((int)sagebwd_workspace_bytes(1, 1, 17, 96), 0, "sagebwd workspace, D = 96");
    expect(sagebwd_workspace_layout(1, 1, 17, 64, NULL), SAGE_FP4_EINVAL, "sagebwd layout, no output");
    void *w = P(0x100000);
    expect(sagebwd_fwd(P(0x1000), P(0x2000), P(0x3000), P(0x4000), (float *)P(0x5000), 2, 3, 300, 64, 2, 0.125f,
                       w, sb, NULL),
           SAGE_FP4_EINVAL, "sagebwd_fwd causal = 2");
    expect(sagebwd_fwd(P(0x1000), P(0x2000), P(0x3000), P(0x4000), (float *)P(0x5000), 2, 3, 300, 64, 0, -1.0f, w,
                       sb, NULL),
           SAGE_FP4_EINVAL, "sagebwd_fwd scale < 0");
    expect(sagebwd_fwd(P(0x1000), P(0x2000), P(0x3000), P(0x4000), (float *)P(0x5000), 2, 3, 300, 64, 0, 0.125f, w,
                       sb - 1, NULL),
           SAGE_FP4_EINVAL, "sagebwd_fwd short workspace");
    expect(sagebwd_bwd(P(0x1000), P(0x2000), (float *)P(0x3000), P(0x4008), P(0x5000), P(0x6000), 2, 3, 300, 64, 0,
                       0.125f, w, sb, NULL),
           SAGE_FP4_EINVAL, "sagebwd_bwd misaligned dq");
    expect(sagebwd_attn_bwd(P(0x1000), P(0x2000), 2, 3, 300, 64, 1, 0.125f, P(0x100010), sb, NULL), SAGE_FP4_EINVAL,
           "sagebwd_attn_bwd misaligned workspace");
    expect(sagebwd_quantize_qkv(P(0x1000), P(0x2000), P(0x3000), 0, 3, 300, 64, w,
                                sagebwd_workspace_bytes(0, 3, 300, 64), NULL),
           SAGE_FP4_OK, "sagebwd empty problem");
    expect(sagebwd_stall_test(0, P(0x1000), P(0x2000), 2, 3, 300, 64, 0.125f, 10, w, sb, NULL), SAGE_FP4_EINVAL,
           "sagebwd stall test, limit too short");
    expect(sagebwd_int_mma_probe((const int8_t *)P(0x1000), (const int8_t *)P(0x2000), 20, (float *)P(0x3000), NULL),
           SAGE_FP4_EINVAL, "sagebwd probe K = 20");
    expect(sagebwd_mma_peak(7, 1, 1, P(0x1000), NULL), SAGE_FP4_EINVAL, "sagebwd peak kind");
    expect(sagebwd_mma_peak(2, 1, (1 << 20) + 1, P(0x1000), NULL), SAGE_FP4_EINVAL, "sagebwd peak iterations");
    expect(sagebwd_umma_probe((const uint16_t *)P(0x1000), (const uint16_t *)P(0x2000), 96, (float *)P(0x3000),
                              (int32_t *)P(0x4000), NULL),
           SAGE_FP4_EINVAL, "sagebwd tcgen05 probe N = 96");
    expect(sagebwd_umma_mn_probe((const uint16_t *)P(0x1001), (const uint16_t *)P(0x2000), (float *)P(0x3000),
                                 (int32_t *)P(0x4000), NULL),
           SAGE_FP4_EINVAL, "sagebwd MN-major probe misaligned a");
    expect(sagebwd_umma_ta_probe((const uint16_t *)P(0x1000), (const uint16_t *)P(0x2008), 64, (float *)P(0x3000),
                                 (int32_t *)P(0x4000), NULL),
           SAGE_FP4_EINVAL, "sagebwd tensor-memory probe misaligned b");
  }

  /* every status code has a string */
  for (int c = -8; c <= 1; c++)
    if (!sage_fp4_strerror(c) || !strlen(sage_fp4_strerror(c))) expect(c, 99, "strerror");
  free(buf);
  if (failures) return 1;
  printf("abi driver: ok\n");
  return 0;
}

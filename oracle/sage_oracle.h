/*
 * sage_oracle.h -- CPU oracle for SageAttention3's microscaled FP4 attention
 * forward.  TEST INFRASTRUCTURE ONLY: tests, the smoke check and the bench's
 * CPU-baseline leg call it; the product library never links or calls it.
 *
 * Plain C, double precision where the method does not fix a precision.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Sources (page, section):
 *   [NEWS-OBST]  senqingzn.com article on SageAttention3, section
 *                "Solving two obstacles and one difficulty": FP4 has only 15
 *                representable values; P lies in [0,1]; 1x16 microscaling for
 *                QK^T and PV; two-level P quantization, per token into
 *                [0, 448*6], then FP4 microscaling.
 *   [NEWS-HW]    same article, section "FP4 attention inference acceleration
 *                and hardware implementation/optimisation": NVFP4 = E2M1 codes,
 *                1x16 blocks, E4M3 scale; FP32 accumulator; the 16-element
 *                max per row is fused with the online softmax row max.
 *   [ABSTRACT]   "SageAttention3: Microscaling FP4 Attention for Inference and
 *                An Exploration of 8-Bit Training", abstract (fugumt.com and
 *                chatpaper.ai copies): FP4 tensor cores accelerate attention,
 *                plug-and-play.
 *
 * Layouts used by the oracle (its own, plain row-major):
 *   Q, K codes   [BH][N_pad][D/2]   element 2i in the low nibble of byte i
 *   Q, K scales  [BH][N_pad][D/16]  one E4M3 byte per 16 elements along D
 *   V^T codes    [BH][D][N_pad/2]   groups run along tokens
 *   V^T scales   [BH][D][N_pad/16]
 * with N_pad = N rounded up to a multiple of 128; padding rows/tokens are 0.
 */
#ifndef SAGE_ORACLE_H
#define SAGE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* codecs */
double sor_e2m1_value(int code);
int sor_e2m1_encode(float x);
double sor_e4m3_value(int bits);
int sor_e4m3_encode(float x);
/* encode the floats whose bit patterns are first .. first+count-1 */
void sor_encode_range(uint32_t first, uint32_t count, uint8_t *e2m1, uint8_t *e4m3);

/* one 16-element group: scale = E4M3(amax/6), codes = E2M1(x * (1/scale)) */
void sor_quant_group16(const float *x, uint8_t *codes16, uint8_t *scale);

/* Microscaling formats: NVFP4 (1x16, E4M3 scales; the method's) and MXFP4
 * (1x32, E8M0 scales; the alternative the pages weighed, [NEWS-HW]). */
#define SOR_FMT_NVFP4 0
#define SOR_FMT_MXFP4 1

/* E8M0 byte -> 2^(b-127); 0xFF is NaN */
double sor_e8m0_value(int b);
/* 32 floats -> 32 E2M1 codes + one E8M0 scale byte (OCP MX rule, see .c) */
void sor_quant_group32_mx(const float *x, uint8_t *codes32, uint8_t *scale);
/* Q/K rows and V in either format (plain layouts as below, with D/32 or
 * N_pad/32 scales per row for MXFP4) */
void sor_quantize_rows_fmt(const uint16_t *x, int BH, int N, int D, int fmt, uint8_t *codes,
                           uint8_t *scales);
void sor_quantize_v_fmt(const uint16_t *v, int BH, int N, int D, int fmt, uint8_t *codes,
                        uint8_t *scales);

/* Q/K rows: bf16 bits [BH][N][D] -> codes/scales as above */
void sor_quantize_rows(const uint16_t *x, int BH, int N, int D, uint8_t *codes, uint8_t *scales);
/* V: bf16 bits [BH][N][D] -> V^T codes/scales, groups along tokens */
void sor_quantize_v(const uint16_t *v, int BH, int N, int D, uint8_t *codes, uint8_t *scales);

/* Tiled FP4 attention over the quantized tensors, softmax scale `scale`
 * (> 0; 1/sqrt(D) is the standard one).
 * fmt: SOR_FMT_NVFP4 or SOR_FMT_MXFP4 (operands quantized in that format).
 * pmode 0 = TILE (level 1 normalises each KV tile's row segment so that its
 * max is 448*6, or 6 for MXFP4), pmode 1 = RUNNING (normalised against the running row max).
 * rows: flat row ids bh*N + i (NULL = all BH*N rows).  out: [nrows][D]. */
int sor_attention(const uint8_t *qc, const uint8_t *qs, const uint8_t *kc, const uint8_t *ks,
                  const uint8_t *vc, const uint8_t *vs, int BH, int N, int D, int causal,
                  int fmt, double scale, int pmode, int kv_tile, const int64_t *rows,
                  int64_t nrows, double *out, double *out_l, double *out_m);

/* sor_attention with the normaliser chosen: lnorm 0 = l from the unquantized
 * probabilities (the method's reading; sor_attention), lnorm 1 = l from the
 * rounded probabilities that enter PV (Direct-P, the rit.work summary of
 * "Hardware-Aware FP4 FlashAttention-4"). */
int sor_attention_ex(const uint8_t *qc, const uint8_t *qs, const uint8_t *kc, const uint8_t *ks,
                     const uint8_t *vc, const uint8_t *vs, int BH, int N, int D, int causal,
                     int fmt, double scale, int pmode, int lnorm, int kv_tile, const int64_t *rows,
                     int64_t nrows, double *out, double *out_l, double *out_m);

/* Exact attention softmax(scale * Q K^T) V, unquantized, from the bf16
 * inputs, in double. */
int sor_attention_exact(const uint16_t *q, const uint16_t *k, const uint16_t *v, int BH, int N,
                        int D, int causal, double scale, const int64_t *rows, int64_t nrows,
                        double *out);

int sor_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif

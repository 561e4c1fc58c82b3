/* sagebwd_oracle.h -- CPU oracle for SageBwd (8-bit attention for training).
 * TEST INFRASTRUCTURE ONLY.  See sagebwd_oracle.c for the method and the
 * readings it follows. */
#ifndef SAGEBWD_ORACLE_H
#define SAGEBWD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The INT8 code of x in a block whose largest magnitude is amax, and the
 * block's dequantization scale amax / 127. */
int sbo_int8_code(float x, float amax);
float sbo_int8_scale(float amax);

/* bf16 bits [BH][N][D] -> INT8 codes [BH][N][D] and one float scale per
 * (head, 128-token block): scales [BH][ceil(N / 128)]. */
void sbo_quantize_blocks(const uint16_t *x, int BH, int N, int D, int8_t *codes, float *scales);

/* Forward and backward of attention with softmax scale `scale` on bf16 q, k,
 * v and the output gradient dout ([BH][N][D] each).  Writes o, the row
 * log-sum-exp lse [BH][N], and dq, dk, dv ([BH][N][D], double).  quant = 1:
 * SageBwd's INT8 and FP16 products; quant = 0: exact float64 attention and
 * its exact gradient.  Returns 0, -1 for invalid arguments (N < 1, D outside
 * [1, 4096], a scale that is not positive and finite), -2 if memory ran out. */
int sbo_attention_train(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                        int BH, int N, int D, int causal, double scale, int quant, double *o,
                        double *lse, double *dq, double *dk, double *dv);

#ifdef __cplusplus
}
#endif
#endif

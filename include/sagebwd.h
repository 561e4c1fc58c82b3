/* sagebwd.h -- C ABI of SageBwd, the 8-bit attention for training, on
 * sm_103a (libsagefp4.so).
 *
 * The method: the senqingzn.com article on SageAttention3, "INT8 attention
 * for training" (six of the seven matrix products of attention's forward and
 * backward passes run in INT8) and "Solving two obstacles and one
 * difficulty", difficulty 3 (the attention-map gradient accumulates
 * quantization error, so the most precision-sensitive backward product stays
 * at FP16); the abstract of "SageAttention3: Microscaling FP4 Attention for
 * Inference and An Exploration of 8-Bit Training" (an 8-bit attention for
 * both forward and backward propagation).
 *
 * What the library computes (the pages leave the granularity open; these
 * are the readings the kernels and the test oracle share):
 *   forward   S = Q^ K^^T (INT8), FlashAttention's online softmax over key
 *             tiles of 128 with the tile probabilities P~ = exp(scale*S - m)
 *             quantized to INT8 per block of 64 queries x 128 keys,
 *             O = sum P~^ V^ / l (INT8 product, l from the unquantized P~);
 *             saves L = log-sum-exp per row.
 *   backward  P = exp(scale*S - L); dV = P^^T dO^ (INT8); dP = dO V^T (FP16
 *             operands, FP32 accumulation); D = rowsum(dO o O);
 *             dS = P o (dP - D); dQ = scale dS^ K^, dK = scale dS^^T Q^ (INT8,
 *             dS quantized per block of 64 queries x 128 keys).
 *   INT8      symmetric per block: scale = amax / 127, code =
 *             rint(x * (127 / amax)) in float arithmetic.  Q, K, V and dO are
 *             quantized per head in blocks of 128 tokens over all D channels.
 *             Inside the attention kernels P's and dS's codes round the exact
 *             product x * (127 / amax) (one fused multiply-add); that differs
 *             from rounding the FP32 product only when the product lies within
 *             half an FP32 unit in the last place of a half-integer.
 *             The INT8 products run on the FP16 tensor path with the codes
 *             held as FP16 values: integer codes, exact products and exact
 *             integer sums (below 2^24), the results of an INT8 MMA, at the
 *             FP16 rate (sm_103a's INT8 MMA runs at a quarter of it;
 *             sagebwd_int_mma_probe checks the exactness on the device).
 *   causal    key j is visible from query i when j <= i.
 *
 * Tensors: q, k, v, o, dout, dq, dk, dv are bf16, contiguous [B][H][N][D],
 * 16-byte aligned, on the current device; lse is float [B][H][N], 4-byte
 * aligned.  D is 64 or 128; N >= 0 (N = 0 or B*H = 0 is a successful no-op).
 * scale is the softmax scale (positive, finite).
 *
 * Workspace: caller-owned device memory of sagebwd_workspace_bytes(B, H, N, D)
 * bytes, 256-byte aligned.  sagebwd_fwd writes the quantized Q, K, V there;
 * sagebwd_bwd reads them back (with the forward's o and lse) and uses the rest
 * as scratch, so the same workspace, untouched in between, must be passed to
 * the backward of the same forward.  Calls on one workspace must be ordered
 * (one stream, or events); the library allocates nothing.
 *
 * Errors: return values are the SAGE_FP4_* codes of sage_fp4.h.  Argument
 * errors (SAGE_FP4_EINVAL) are found before anything touches the device;
 * SAGE_FP4_EUNSUPPORTED on a device other than sm_103; SAGE_FP4_ECUDA when a
 * launch fails.  The kernels run asynchronously on `stream` (a cudaStream_t,
 * NULL for the legacy default stream); a copy that never completes makes the
 * kernels give up after 1.5 s and record SAGE_FP4_ETIMEOUT in the
 * workspace's status word, which sagebwd_get_status reads.
 */
#ifndef SAGEBWD_H
#define SAGEBWD_H

#include <stddef.h>
#include <stdint.h>

#include "sage_fp4.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Number of regions in the workspace (see sagebwd_workspace_layout). */
#define SAGEBWD_WS_FIELDS 17

/* Bytes of workspace for these sizes; 0 when the sizes are invalid. */
size_t sagebwd_workspace_bytes(int B, int H, int N, int D);

/* Byte offsets of the workspace's regions, in this order: the INT8 codes of
 * Q, K, V, dO (as FP16 values), V and dO as FP16 (each [B*H][N padded to
 * 128][D], the 16-byte chunks of row r XOR-permuted by r & 7); the codes of Q,
 * dO and V transposed per 64-token tile ([B*H][N/64][D][64], swizzled the
 * same way); the Q/K/V/dO
 * block scales (float [B*H][ceil(N/128)] each); -L in log2 units and
 * D = rowsum(dO o O) (float [B*H][N padded to 128]); the dQ accumulator
 * (float [B*H][N padded][D]); the status word.  For tests and inspection;
 * offsets must hold SAGEBWD_WS_FIELDS values. */
int sagebwd_workspace_layout(int B, int H, int N, int D, size_t *offsets);

/* Forward: quantizes q, k, v into the workspace and writes o (bf16) and lse
 * (natural-log log-sum-exp of scale * S per row).  The same as
 * sagebwd_quantize_qkv followed by sagebwd_attn_fwd. */
int sagebwd_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N, int D,
                int causal, float scale, void *workspace, size_t workspace_bytes, void *stream);

/* Backward: given dout and the forward's o and lse (and its workspace),
 * writes dq, dk, dv (bf16).  The same as sagebwd_bwd_prep, sagebwd_attn_bwd
 * and sagebwd_dq_out in turn. */
int sagebwd_bwd(const void *dout, const void *o, const float *lse, void *dq, void *dk, void *dv, int B, int H,
                int N, int D, int causal, float scale, void *workspace, size_t workspace_bytes, void *stream);

/* The steps, one kernel launch each, on the same arguments and workspace:
 *   quantize_qkv  Q, K, V -> INT8 codes and block scales, and V as FP16;
 *   attn_fwd      the forward attention from those codes -> o, lse;
 *   bwd_prep      dO -> codes, scales and FP16 copy; D = rowsum(dout o o);
 *                 L from lse; zeroes the dQ accumulator;
 *   attn_bwd      dK, dV (bf16), and dQ into the FP32 accumulator;
 *   dq_out        the accumulator -> dq (bf16). */
int sagebwd_quantize_qkv(const void *q, const void *k, const void *v, int B, int H, int N, int D, void *workspace,
                         size_t workspace_bytes, void *stream);
int sagebwd_attn_fwd(void *o, float *lse, int B, int H, int N, int D, int causal, float scale, void *workspace,
                     size_t workspace_bytes, void *stream);
int sagebwd_bwd_prep(const void *dout, const void *o, const float *lse, int B, int H, int N, int D, void *workspace,
                     size_t workspace_bytes, void *stream);
int sagebwd_attn_bwd(void *dk, void *dv, int B, int H, int N, int D, int causal, float scale, void *workspace,
                     size_t workspace_bytes, void *stream);
int sagebwd_dq_out(void *dq, int B, int H, int N, int D, void *workspace, size_t workspace_bytes, void *stream);

/* Synchronizes `stream`, returns the workspace's status word (0 or a
 * negative SAGE_FP4_* code) and clears it. */
int sagebwd_get_status(void *workspace, int B, int H, int N, int D, void *stream);

/* Throughput probe of the MMA forms the kernels use.  Kinds 0 and 1: warp-level
 * MMAs on register operands, INT8 m16n8k32 and FP16 m16n8k16 with FP32
 * accumulation; each of `ctas` CTAs of 256 threads runs iters x 8 MMAs per
 * warp.  Kinds 2, 3, 4: tcgen05.mma kind::f16 with M = 128, K = 16 and N = 64,
 * 128, 256 (K-major shared-memory operands, FP32 accumulation in tensor
 * memory); kind 5: N = 64 with A in tensor memory; kind 6: N = 64 with B
 * MN-major.  One thread of each of `ctas` CTAs issues iters x 8 of them
 * (iters <= 2^20).
 * scratch is 4 device bytes it may write (SAGE_FP4_ETIMEOUT when a tcgen05
 * completion wait runs out). */
int sagebwd_mma_peak(int kind, int ctas, int iters, void *scratch, void *stream);

/* Failure-detection test: runs the forward attention (kernel 0; out0 = o,
 * out1 = lse) or the backward attention (kernel 1; out0 = dk, out1 = dv),
 * non-causal, on a workspace already filled by sagebwd_quantize_qkv (and, for
 * kernel 1, sagebwd_bwd_prep), with one copy withheld: the first CTA never
 * issues its first streamed tile, so its bounded wait runs out after
 * wait_limit_ns (1 ms to 1.5 s) and the kernel records SAGE_FP4_ETIMEOUT in
 * the status word; every other CTA completes.  The outputs are then
 * incomplete.  EINVAL for an empty problem. */
int sagebwd_stall_test(int kernel, void *out0, void *out1, int B, int H, int N, int D, float scale,
                       uint64_t wait_limit_ns, void *workspace, size_t workspace_bytes, void *stream);

/* Probe of the 5th-generation tensor-core form the backward uses (tcgen05.mma
 * kind::f16 with the 128-byte-swizzled K-major operand layout): one CTA
 * computes c [128][N] = a [128][64] x b [N][64]^T (FP16 in, FP32 out; all
 * row-major device arrays; N = 64 or 128).  status: a device int32 that a
 * wait that runs out sets to SAGE_FP4_ETIMEOUT. */
int sagebwd_umma_probe(const uint16_t *a, const uint16_t *b, int N, float *c, int32_t *status, void *stream);

/* Probe of the tensor-memory A operand (tcgen05.mma kind::f16 with A written to
 * tensor memory by tcgen05.st, 128 rows in lanes, two FP16 values per 32-bit
 * column, the lower K index in the low half; B 128-byte-swizzled K-major in
 * shared memory): one CTA computes c [128][N] = a [128][64] x b [N][64]^T
 * (FP16 in, FP32 out; row-major device arrays; N = 64 or 128).  status: a
 * device int32 that a wait that runs out sets to SAGE_FP4_ETIMEOUT. */
int sagebwd_umma_ta_probe(const uint16_t *a, const uint16_t *b, int N, float *c, int32_t *status, void *stream);

/* Probe of the MN-major operand form dQ = dS^ K^ uses (tcgen05.mma kind::f16,
 * both operands stored with the K index as the 128-byte row, A's two 64-row
 * blocks of M 32 KB apart): one CTA computes c [128][64] = a [128][128] x
 * b [128][64] (FP16 in, FP32 out; row-major device arrays).  status: a device
 * int32 that a wait that runs out sets to SAGE_FP4_ETIMEOUT. */
int sagebwd_umma_mn_probe(const uint16_t *a, const uint16_t *b, float *c, int32_t *status, void *stream);

/* Exactness probe of the INT8 products: the 16 x 8 product of INT8 device
 * matrices a [16][K] and b [8][K] (row-major, K a multiple of 16 up to 4096)
 * computed the kernels' way (codes as FP16 values, FP32 accumulation chained
 * over K/16 MMAs), written to out, float [16][8] on the device. */
int sagebwd_int_mma_probe(const int8_t *a, const int8_t *b, int K, float *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif

/*
 * sage_fp4.h -- C ABI of the GB300 (sm_103a) NVFP4 attention forward library.
 *
 * The method is SageAttention3's microscaled FP4 attention for inference:
 *   - Q, K and V are quantized to NVFP4: E2M1 4-bit codes with one E4M3 scale
 *     per 1x16 group (senqingzn.com article on SageAttention3, section
 *     "Solving two obstacles and one difficulty", solution 1; section "FP4
 *     attention inference acceleration and hardware implementation/
 *     optimisation", NVFP4 paragraph);
 *   - S = Q K^T and O = P V run on FP4 tensor cores with FP32 accumulation
 *     (same section, accumulator paragraph; abstract of "SageAttention3:
 *     Microscaling FP4 Attention for Inference and An Exploration of 8-Bit
 *     Training");
 *   - the online softmax is fused with a two-level quantization of P: each
 *     token's row segment is first rescaled into [0, 448*6], then quantized
 *     to NVFP4 in 1x16 groups (section "Solving two obstacles and one
 *     difficulty", solution 2; the 16-element row maximum is fused with the
 *     online softmax, hardware section).
 *
 * Conventions for every call:
 *   - B, H, N, D: batch, heads, sequence length, head dimension.  D is 64 or
 *     128.  Q, K, V and O are bf16, contiguous [B, H, N, D].
 *   - N_pad = N rounded up to a multiple of 128.
 *   - The softmax scale is 1/sqrt(D).  Causal: key j is visible to query i
 *     iff j <= i (queries and keys share one sequence).
 *   - Every pointer passed to a computing call is DEVICE memory owned by the
 *     caller, except the q, k, v, o of sage_fp4_attention_host (host memory).
 *     The library allocates no memory, frees nothing and keeps no global state
 *     besides per-device caches of kernel attributes and, once
 *     sage_fp4_attention_host has run on a device, that call's three streams
 *     and ten events.  All computing calls are asynchronous on `stream` (a
 *     cudaStream_t; NULL = legacy default stream).
 *   - Inputs must be finite; NaN or Inf inputs give unspecified results.
 *   - Return value: SAGE_FP4_OK or a negative status.  Argument errors are
 *     detected on the host before anything is launched.  Errors found while a
 *     kernel runs (a bounded wait that gave up) are written to the status word
 *     and returned by sage_fp4_get_status().
 *
 * NVFP4 tensor layout (one quantized operand):
 *   codes   packed E2M1, two per byte, the element with the even index in the
 *           LOW nibble.  E2M1: bit 3 sign, bits 2-1 exponent (bias 1), bit 0
 *           mantissa; values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives.
 *   scales  E4M3 (bias 7, largest 448, sign bit 0), one per 16 elements along
 *           the operand's contraction axis, stored in the 128x4 block layout
 *           that block-scaled tensor-core MMAs read: for an operand of R rows
 *           (R padded to a multiple of 128) and C contraction elements (C a
 *           multiple of 64), the scale of row r and group g (g = element/16)
 *           is at byte
 *             ((r/128) * (C/64) + g/4) * 512 + (r%32) * 16 + ((r%128)/32) * 4 + g%4.
 *   q, k    rows are tokens: codes [B*H][N_pad][D/2], scales with R = N_pad,
 *           C = D, per (b,h) N_pad*D/16 bytes.  Groups run along D.
 *   vt      V transposed, rows are channels: codes [B*H][D][N_pad/2], scales
 *           with R = 128 (D padded to 128), C = N_pad, per (b,h) 8*N_pad bytes.
 *           Groups run along tokens, the contraction axis of P V.
 *   Rows/tokens in [N, N_pad) and padding channel rows hold code 0, scale 0.
 *
 * Quantization rule for one group x[0..15] (the pages fix the format, not the
 * rounding; this is the reading, identical in the CPU oracle):
 *   s = E4M3_rn(amax/6), with amax/6 a round-to-nearest float division;
 *   if s == 0 every code is 0; else r = 1/s (round-to-nearest float) and
 *   code_i = E2M1_rn(x_i * r) with the product rounded to float once;
 *   both conversions round to nearest, ties to even, and saturate (E2M1 at
 *   +-6, E4M3 at 448); a negative value that rounds to zero is -0 (code 0x8).
 */
#ifndef SAGE_FP4_H
#define SAGE_FP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SAGE_FP4_OK 0
#define SAGE_FP4_EINVAL (-1)      /* bad argument: null or misaligned pointer, bad size or D */
#define SAGE_FP4_ECUDA (-2)       /* CUDA runtime/driver error at launch or copy */
#define SAGE_FP4_ETIMEOUT (-3)    /* a kernel's bounded wait gave up (see sage_fp4_get_status) */
#define SAGE_FP4_EUNSUPPORTED (-4) /* device is not sm_103 (the kernels are built for sm_103a) */
#define SAGE_FP4_ETOOLARGE (-5)
/* debug build only (SAGE_FP4_DEBUG_BOUNDS=1, libsagefp4_debug.so): a kernel
 * computed a global-memory index outside its buffer; the access was skipped */
#define SAGE_FP4_EBOUNDS (-6)   /* problem needs more than the no-allocation entry's fixed scratch */

/* Microscaling formats of the quantized operands.  NVFP4 is the method's:
 * E2M1 codes with one E4M3 scale per 16 elements.  MXFP4 is the alternative
 * the pages weighed and set aside for accuracy ([NEWS-HW] data-type
 * paragraph): E2M1 codes with one E8M0 scale (a power of two, 2^(b-127)) per
 * 32 elements.  Scale rule for an MXFP4 group (the OCP MX v1.0 conversion;
 * the pages fix only the format): b = max(exponent field of amax - 2, 0),
 * code_i = E2M1_rn(x_i * 2^(127-b)), saturating.  MXFP4 operands use the
 * same layouts and sizes as NVFP4: in each 32-bit scale word of the block
 * layout (one per row and K = 64 step) bytes 0 and 1 hold the step's two E8M0
 * scales and bytes 2 and 3 are zero.  In attention, P is quantized in the
 * same format; its first level then normalises each row segment's maximum
 * to 6 instead of 448*6 (E8M0 needs no range help, and 6 keeps the maximum
 * exact). */
#define SAGE_FP4_FORMAT_NVFP4 0
#define SAGE_FP4_FORMAT_MXFP4 1
/* Direct-P (the rit.work summary of "Hardware-Aware FP4 FlashAttention-4",
 * "Что сделали"): MXFP4 operands and P as SAGE_FP4_FORMAT_MXFP4, but the
 * softmax normaliser l is summed from the rounded P (decoded codes times
 * their scales, the values PV uses) instead of from the unquantized
 * exponentials.  Quantization treats it as SAGE_FP4_FORMAT_MXFP4;
 * sage_fp4_attn_fwd_ex takes it with contiguous O only (SAGE_FP4_EINVAL for
 * other strides). */
#define SAGE_FP4_FORMAT_MXFP4_DIRECTP 2

typedef struct sage_fp4_tensor {
  uint8_t *codes;  /* packed E2M1, 16-byte aligned */
  uint8_t *scales; /* E4M3 in the 128x4 block layout, 16-byte aligned */
} sage_fp4_tensor;

typedef struct sage_fp4_qkv {
  sage_fp4_tensor q;  /* quantized Q, rows = tokens */
  sage_fp4_tensor k;  /* quantized K, rows = tokens */
  sage_fp4_tensor vt; /* quantized V^T, rows = channels */
  int32_t *status;    /* one int32 in device memory, zero-initialised by the caller */
} sage_fp4_qkv;

/* Element strides of a bf16 [B,H,N,D] tensor whose D axis is contiguous:
 * element (b, h, n, d) is at b*b_stride + h*h_stride + n*n_stride + d.  Each
 * stride is >= 0 and a multiple of 8 (16 bytes).  Calls that take a pointer
 * to strides read NULL as the contiguous [B,H,N,D] layout; [B,N,H,D] (NHD) is
 * {N*H*D, D, H*D}; Q of a packed [B,N,3,H,D] QKV tensor is {3*N*H*D, D, 3*H*D}. */
typedef struct sage_fp4_strides {
  int64_t b, h, n;
} sage_fp4_strides;

/* Bytes of one device buffer that holds all quantized operands plus the status
 * word, each sub-buffer 256-byte aligned.  0 if the sizes are invalid. */
size_t sage_fp4_workspace_bytes(int B, int H, int N, int D);

/* Carve `workspace` (device memory of at least sage_fp4_workspace_bytes bytes,
 * 256-byte aligned) into the operand pointers of *out.  Pointer arithmetic
 * only: nothing is launched, nothing is written to the device.  The status
 * word must still be zeroed by the caller (e.g. by zeroing the workspace). */
int sage_fp4_qkv_from_workspace(void *workspace, size_t workspace_bytes, int B, int H, int N,
                                int D, sage_fp4_qkv *out);

/* Quantize bf16 Q, K, V ([B,H,N,D], contiguous, 16-byte aligned device memory)
 * into the NVFP4 operands of *out (layouts above): Q and K along D, V along
 * tokens into V^T.  Codes and scales are bit-exact with the rule above.
 * Two kernel launches on `stream`; the second (V) is a programmatic dependent of
 * the first and may start while the first drains, and it completes only after
 * the first, so work queued after this call sees both.  out->status
 * (zero-initialised) is set to SAGE_FP4_ETIMEOUT if a bounded device wait for
 * a tile copy gives up. */
int sage_fp4_quantize_qkv(const void *q, const void *k, const void *v, const sage_fp4_qkv *out,
                          int B, int H, int N, int D, void *stream);

/* sage_fp4_quantize_qkv for inputs in any layout with a contiguous D axis:
 * q, k and v each with its own strides (NULL = contiguous [B,H,N,D]); 16-byte
 * aligned device memory.  The quantized operands are the same as for the
 * contiguous copies of the inputs, bit for bit.  format: SAGE_FP4_FORMAT_NVFP4
 * (as sage_fp4_quantize_qkv) or SAGE_FP4_FORMAT_MXFP4.  SAGE_FP4_EINVAL for
 * another format, a negative or unaligned stride, or offsets beyond 2^62
 * elements.  No
 * counterpart in the pages, which describe no API (the plug-and-play use of
 * the abstract). */
int sage_fp4_quantize_qkv_strided(const void *q, const sage_fp4_strides *q_strides, const void *k,
                                  const sage_fp4_strides *k_strides, const void *v,
                                  const sage_fp4_strides *v_strides, const sage_fp4_qkv *out,
                                  int B, int H, int N, int D, int format, void *stream);

/* Attention forward over quantized operands: O = softmax(Q K^T / sqrt(D)) V
 * computed by the SageAttention3 FP4 method (block-scaled FP4 MMAs with FP32
 * accumulation; online softmax over KV tiles of 128 keys fused with two-level
 * P quantization, level 1 normalising each KV tile's row segment so that its
 * maximum becomes 448*6).  o: bf16 [B,H,N,D] device memory, written in full.
 * One kernel launch on `stream`.  Kernel-time failures set *qkv->status. */
int sage_fp4_attn_fwd(const sage_fp4_qkv *qkv, void *o, int B, int H, int N, int D, int causal,
                      void *stream);

/* sage_fp4_attn_fwd with an explicit softmax scale, O = softmax(softmax_scale
 * * Q K^T) V, and O written through o_strides (NULL = contiguous [B,H,N,D];
 * the rows of O must not overlap).  softmax_scale must be > 0 and at most
 * 1e30 (sage_fp4_attn_fwd uses 1/sqrt(D)); anything else is SAGE_FP4_EINVAL.
 * The scale multiplies S before the exponentials of the online softmax and of
 * the first P-quantization level (the pages give the method no scale; this is
 * the one a drop-in attention takes).  format: the format the operands were
 * quantized in (SAGE_FP4_FORMAT_NVFP4 or SAGE_FP4_FORMAT_MXFP4); P is
 * quantized in the same one.  SAGE_FP4_FORMAT_MXFP4_DIRECTP: MXFP4 with the
 * Direct-P normaliser (contiguous O only). */
int sage_fp4_attn_fwd_ex(const sage_fp4_qkv *qkv, void *o, const sage_fp4_strides *o_strides, int B,
                         int H, int N, int D, int causal, float softmax_scale, int format,
                         void *stream);

/* No counterpart in the pages: the failure-detection test of the attention
 * kernel's bounded waits.  The same launch as sage_fp4_attn_fwd, except that
 * the kernel's K-tile producer stops after the first KV tile of each CTA's
 * stream and every bounded wait gives up after wait_limit_ns (1 ms to 1.5 s;
 * sage_fp4_attn_fwd uses 1.5 s).  The waiting roles then abandon their work:
 * copies and tensor-core operations in flight are waited for, tensor memory is
 * freed, nothing faults, and *qkv->status becomes SAGE_FP4_ETIMEOUT.  O is left
 * partly written.  Returns SAGE_FP4_EINVAL for a limit out of range, else as
 * sage_fp4_attn_fwd; read the outcome with sage_fp4_get_status. */
int sage_fp4_attn_fwd_stall_test(const sage_fp4_qkv *qkv, void *o, int B, int H, int N, int D,
                                 int causal, uint64_t wait_limit_ns, void *stream);

/* No counterpart in the pages: the failure-detection test of the V
 * quantizer's bounded waits.  The same launch as sage_fp4_quantize_qkv,
 * except that one block of the V kernel never issues the copy of its first
 * tile and every wait for a tile gives up after wait_limit_ns (1 ms to 1.5 s;
 * sage_fp4_quantize_qkv uses 1.5 s).  That block then leaves as a whole, after
 * the copies it still has in flight have landed; nothing faults, and
 * *out->status becomes SAGE_FP4_ETIMEOUT.  The V^T operands are left partly
 * written.  Returns SAGE_FP4_EINVAL for a limit out of range, else as
 * sage_fp4_quantize_qkv; read the outcome with sage_fp4_get_status. */
int sage_fp4_quantize_qkv_stall_test(const void *q, const void *k, const void *v,
                                     const sage_fp4_qkv *out, int B, int H, int N, int D,
                                     uint64_t wait_limit_ns, void *stream);

/* Synchronise `stream`, read the status word of `qkv`, reset it to 0 and
 * return it (SAGE_FP4_OK, SAGE_FP4_ETIMEOUT) or SAGE_FP4_ECUDA if the copy
 * itself failed. */
int sage_fp4_get_status(const sage_fp4_qkv *qkv, void *stream);

/* Static description of a status code. */
const char *sage_fp4_strerror(int status);

/* ---- one-call attention for callers that cannot allocate ------------------ */

/* Size of the fixed device scratch array behind sage_fp4_attention_noalloc. */
#define SAGE_FP4_NOALLOC_SCRATCH_BYTES (64u << 20)

/* No counterpart in the pages: a convenience of this library.  Quantize bf16
 * q, k, v ([B,H,N,D], contiguous, 16-byte aligned) and run the attention
 * forward into bf16 o, in one call that allocates nothing.  It is meant for
 * callers that cannot call cudaMalloc: code running inside another
 * framework's operator without access to its allocator, plugins whose host
 * owns every device allocation, code that must not allocate after start-up.
 *
 * The call is sage_fp4_quantize_qkv followed by sage_fp4_attn_fwd over a
 * workspace carved from one file-scope device array of
 * SAGE_FP4_NOALLOC_SCRATCH_BYTES (64 MiB), with the caller's status word in
 * place of the workspace's; their argument checks and results apply
 * unchanged.  Every GPU that loads the library's module holds that array
 * until the process exits.  Problems whose workspace
 * (sage_fp4_workspace_bytes) exceeds the array are rejected with
 * SAGE_FP4_ETOOLARGE before anything runs; the LLM prefill shape B1 H32 N8192
 * D128 (~54 MiB) fits, B4 H32 N4096 D128 (~108 MiB) does not.
 *
 * status: one int32 of device memory, zero-initialised by the caller, set to
 * SAGE_FP4_ETIMEOUT if a bounded device wait gives up (as in
 * sage_fp4_attn_fwd; launches skip their work while it is nonzero).
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and keeps it, keyed by the current CUDA context's
 * unique ID, so that a context created after cudaDeviceReset, or a second
 * context on the device, gets a lookup of its own; make that first call
 * before any stream capture.  All calls share the array and it keeps the last
 * call's contents;
 * each call rewrites every byte it reads, so nothing has to be cleared
 * between calls.  Calls whose work overlaps on the GPU (unordered streams or
 * host threads) race on the array: order them.  Asynchronous on `stream`;
 * three kernel launches. */
int sage_fp4_attention_noalloc(const void *q, const void *k, const void *v, void *o,
                               int32_t *status, int B, int H, int N, int D, int causal,
                               void *stream);

/* ---- the whole path from host memory -------------------------------------- */

/* Bytes of device workspace sage_fp4_attention_host needs for this problem
 * (0 if the sizes are invalid).  About 3 * (4 * c * N * D * 2) bytes plus
 * three sets of quantized operands, c = ceil(B*H / 8) heads per chunk. */
size_t sage_fp4_host_workspace_bytes(int B, int H, int N, int D);

/* No counterpart in the pages: a convenience of this library for callers
 * whose tensors live in host memory.  The same result as
 * sage_fp4_quantize_qkv followed by sage_fp4_attn_fwd (bit-identical O), with
 * q, k, v (bf16 [B,H,N,D], contiguous) read from host memory and o written to
 * host memory.  Page-locked (pinned) host memory lets the copies overlap the
 * kernels; pageable memory works, but its copies do not overlap.
 *
 * The B*H heads are cut into chunks of ceil(B*H / 8) heads and pipelined
 * through three staging slots of `workspace` on three streams of the
 * library's own (copy in / quantize + attention / copy out), so that while
 * chunk i computes, chunk i+1 is copied in and chunk i-1 copied out.  The
 * call forks from `stream` (the pipeline starts after the work queued on
 * `stream` before it) and joins back into it (work queued on `stream` after
 * it starts once o is complete in host memory); it is therefore asynchronous
 * like every other call, and usable under stream capture.  Calls on one
 * device are serialised on the host while they enqueue.
 *
 * workspace: device memory of at least sage_fp4_host_workspace_bytes bytes,
 *   256-byte aligned; its contents need no initialisation.  Calls sharing a
 *   workspace must be ordered (one stream, or events).
 * status: one int32 of device memory, zero-initialised by the caller, set to
 *   SAGE_FP4_ETIMEOUT if a kernel's bounded wait gives up (later chunks then
 *   skip their work).
 * Returns SAGE_FP4_EINVAL for bad arguments (checked before anything is
 * queued), SAGE_FP4_ECUDA if queuing a copy, event or kernel failed (work
 * already queued then still runs; synchronise before reusing the buffers). */
int sage_fp4_attention_host(const void *q, const void *k, const void *v, void *o, int B, int H,
                            int N, int D, int causal, void *workspace, size_t workspace_bytes,
                            int32_t *status, void *stream);

/* ---- diagnostics (tests use these to pin the device primitives) ---------- */

/* Convert the floats whose bit patterns are first .. first+count-1 with the
 * device's round-to-nearest saturating conversions used by the kernels:
 * e2m1[i] = E2M1 code (low nibble), e4m3[i] = E4M3 byte.  Either output may
 * be NULL.  Device memory. */
int sage_fp4_cvt_probe(uint32_t first, uint32_t count, uint8_t *e2m1, uint8_t *e4m3,
                       void *stream);

/* One block-scaled FP4 tensor-core product D = A B^T for a 128-row tile, the
 * building block of S = Q K^T and O = P V.  a: codes [128][K/2] and scales
 * (block layout, R = 128, C = K); b: codes [n][K/2] and scales (R = 128 with
 * rows >= n zero, C = K); d: float [128][n] row-major.  K in {64, 128, 256},
 * n in {64, 128}.  a_by_threads = 1 stages A through ordinary shared-memory
 * stores in the kernel's swizzled layout (the path P takes); 0 loads it with
 * the tensor-memory-access engine (the path Q, K, V take).  status: one
 * zero-initialised int32 that a timed-out wait sets to SAGE_FP4_ETIMEOUT.
 * Device memory; codes and scales 16-byte aligned.  One launch on `stream`. */
int sage_fp4_mma_probe(const uint8_t *a_codes, const uint8_t *a_scales, const uint8_t *b_codes,
                       const uint8_t *b_scales, int n, int K, int a_by_threads, float *d,
                       int32_t *status, void *stream);

/* The same product for MXFP4 operands (kind::mxf4: E2M1 codes, one E8M0
 * scale per 32 elements, [NEWS-HW]'s alternative format).  Scales are given as
 * for sage_fp4_mma_probe, 512 bytes per K = 64 step in the block layout's
 * positions: the word of row r holds that row's two E8M0 scales of the step
 * in bytes 0 and 1; bytes 2 and 3 are not read. */
int sage_fp4_mma_probe_mx(const uint8_t *a_codes, const uint8_t *a_scales, const uint8_t *b_codes,
                          const uint8_t *b_scales, int n, int K, int a_by_threads, float *d,
                          int32_t *status, void *stream);

/* sage_fp4_mma_probe / sage_fp4_mma_probe_mx with options as flags:
 *   SAGE_FP4_PROBE_A_BY_THREADS  a_by_threads = 1 above;
 *   SAGE_FP4_PROBE_MX            the MXFP4 product of sage_fp4_mma_probe_mx;
 *   SAGE_FP4_PROBE_SF_ROWS128    A's scale factors reach tensor memory by
 *       128-lane copies (one per two K = 64 steps, or per step when K = 64),
 *       matrix row r to lane r, from a 128-row source that holds row r's scale
 *       word of a step in word r / 32 of the row's 16 bytes and NaN-valued
 *       noise in the other three (B's stay replicated in all four lane
 *       quarters).  The product is exact only if the MMA reads A row r's scales
 *       from lane r, column (step base) + r / 32, and nothing else of those
 *       columns: the layout in which the attention kernel's softmax writes P's
 *       scales.
 * Other bits: SAGE_FP4_EINVAL.  Arguments and errors otherwise as above. */
#define SAGE_FP4_PROBE_A_BY_THREADS 1
#define SAGE_FP4_PROBE_MX 2
#define SAGE_FP4_PROBE_SF_ROWS128 4
int sage_fp4_mma_probe_ex(const uint8_t *a_codes, const uint8_t *a_scales, const uint8_t *b_codes,
                          const uint8_t *b_scales, int n, int K, int flags, float *d,
                          int32_t *status, void *stream);

/* The tensor-core rate of the attention kernel's MMA instruction, for the
 * roofline: one block per SM, each with one thread issuing iters
 * back-to-back block-scaled FP4 MMAs (M = 128, N = n, K = 64, E4M3 scales,
 * kind::mxf4nvf4) on operands in shared memory, then one commit and a bounded
 * wait.  The caller times the launch: FLOPs = 2 * 128 * n * 64 * iters * (number
 * of SMs).  iters 1 .. 10^6, n 128 or 256.  status: one zero-initialised
 * int32, set to SAGE_FP4_ETIMEOUT if the wait gives up.  No counterpart in the
 * pages. */
int sage_fp4_mma_peak(int iters, int n, int32_t *status, void *stream);

/* The reducing tensor-memory load from which the attention kernel takes the
 * 16-key group maxima of a tile row (the fusion of the group maxima with the
 * row maximum, senqingzn.com article, "FP4 attention inference acceleration
 * and hardware implementation/optimisation"): one block of 128 threads stores
 * in[r][c] (FP32, 128 x 128, row-major, r = tensor-memory lane) into tensor
 * memory, reads each row back in eight 16-column groups with
 * tcgen05.ld.red.max, and writes the values read to vals[r][c] and the
 * maximum the instruction reported for group g to maxes[r][g] (128 x 8).
 * All three are device pointers, 16-byte aligned.  No counterpart in the
 * pages. */
int sage_fp4_tmem_max_probe(const float *in, float *vals, float *maxes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SAGE_FP4_H */

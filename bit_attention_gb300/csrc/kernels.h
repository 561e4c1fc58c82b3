// kernels.h -- launchers shared between the kernel translation units and the
// C ABI (api.cu).  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#ifndef SAGE_FP4_DEBUG_BOUNDS
#define SAGE_FP4_DEBUG_BOUNDS 0
#endif

namespace sagefp4 {

// The sizes every computed global-memory index is checked against in the
// debug build (SAGE_FP4_DEBUG_BOUNDS=1); the release build ignores them.
struct Extents {
  int32_t* status;        // where a failed check is recorded (SAGE_FP4_EBOUNDS)
  long long x[3];         // bf16 elements addressable through q, k, v (largest offset + 1)
  long long o;            // bf16 elements addressable through o
  long long codes, scales;          // bytes of one Q or K code / scale buffer
  long long vt_codes, vt_scales;    // bytes of the V^T code / scale buffer
};

// True if [off, off + len) lies in [0, extent).  Debug build: otherwise the
// first failure is recorded in *e.status and the caller skips the access.
// Release build: always true, so the check and its arithmetic compile away.
__device__ __forceinline__ bool in_bounds(const Extents& e, long long off, long long len, long long extent) {
#if SAGE_FP4_DEBUG_BOUNDS
  if (off >= 0 && off + len <= extent) return true;
  atomicCAS(e.status, 0, -6);  // SAGE_FP4_EBOUNDS
  return false;
#else
  (void)e;
  (void)off;
  (void)len;
  (void)extent;
  return true;
#endif
}

// Element strides of a bf16 [B,H,N,D] tensor between batches, heads and
// tokens; D is contiguous.  All three are multiples of 8 (16 bytes).
struct Strides {
  long long b, h, n;
};

// Strides of the contiguous [B,H,N,D] layout.
inline Strides contiguous_bhnd(int H, int N, int D) {
  return Strides{static_cast<long long>(H) * N * D, static_cast<long long>(N) * D, D};
}

// mx: MXFP4 (groups of 32, E8M0 scales) instead of NVFP4.
cudaError_t launch_quant_rows(const void* q, const void* k, Strides sq, Strides sk, uint8_t* qc,
                              uint8_t* qs, uint8_t* kc, uint8_t* ks, int H, int BH, int N, int D,
                              bool mx, const Extents& ext, cudaStream_t st);
// wait_ns bounds every wait for a tile; withhold: failure-detection test (block
// 0 never issues its first tile).
cudaError_t launch_quant_v(const void* v, Strides sv, uint8_t* vc, uint8_t* vs, int H, int BH, int N,
                           int D, bool mx, int32_t* status, uint64_t wait_ns, int withhold,
                           const Extents& ext, cudaStream_t st);

struct AttnParams {
  const uint8_t* sfq;  // Q scales (block layout), per (b,h) N_pad*D/16 bytes
  const uint8_t* sfk;  // K scales
  const uint8_t* sfv;  // V^T scales, per (b,h) 8*N_pad bytes
  void* o;             // bf16 O, row (b, h, n) at element b*os.b + h*os.h + n*os.n
  Strides os;
  int32_t* status;
  int H, BH, N, Np, causal, n_qt;
  float a;  // log2(e) * softmax scale: the scale folded into exp2
  int mx;   // 1: operands are MXFP4 (groups of 32, E8M0 scales), P quantized the same way;
            // 2: the same with the row sum from the rounded P (Direct-P; dense O only)
  int flags;           // kAttnWithholdK: failure-detection test (see below)
  uint64_t wait_ns;    // limit of every bounded wait in the kernel
#if SAGE_FP4_DEBUG_BOUNDS
  Extents ext;         // sizes the scale copies and O stores are checked against
#endif
};

// Failure-detection test: the K producer issues the first KV tile of its
// stream and then stops, so the S issuer's bounded wait for the next tile
// gives up, sets the status word to SAGE_FP4_ETIMEOUT, and every role
// abandons its work through the normal drain path.
constexpr int kAttnWithholdK = 1;
constexpr uint64_t kAttnWaitNs = 1500ull * 1000ull * 1000ull;  // 1.5 s

cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const AttnParams& p, int D, cudaStream_t st);

cudaError_t launch_cvt_probe(uint32_t first, uint32_t count, uint8_t* e2m1, uint8_t* e4m3,
                             cudaStream_t st);

struct MmaProbeParams {
  const uint8_t* a_codes;
  const uint8_t* a_scales;
  const uint8_t* b_scales;
  float* d;
  int32_t* status;
  int n, K, a_by_threads;
  int mx;  // 1: MXFP4 product (kind::mxf4, UE8M0 scales, two per row per K = 64)
  // 1: A's scale factors copied without replication, row r of the matrix to
  // lane r (tcgen05.cp .128x256b per two K = 64 steps, .128x128b for K = 64),
  // from a 128-row source that holds row r's scale word in word r / 32 of its
  // 16 bytes and NaN-valued noise in the other three
  int sf_rows128;
};
cudaError_t launch_mma_probe(const CUtensorMap& ta, const CUtensorMap& tb, const MmaProbeParams& p,
                             cudaStream_t st);
cudaError_t launch_mma_peak(int iters, int n, int32_t* status, cudaStream_t st);
cudaError_t launch_tmem_max_probe(const float* in, float* vals, float* maxes, cudaStream_t st);

}  // namespace sagefp4

// quant.cu -- NVFP4 quantization of Q, K (groups of 16 along D) and V (groups
// of 16 along tokens, written as V^T), bit-exact with the rule in sage_fp4.h.
//
// Method: 1x16 microscaling of both products (senqingzn.com article on
// SageAttention3, "Solving two obstacles and one difficulty", solution 1);
// NVFP4 = E2M1 codes + one E4M3 scale per 16 elements ("FP4 attention
// inference acceleration and hardware implementation/optimisation").
//
// Both kernels are HBM-bound streams: 2 bytes read and 0.5625 bytes written
// per element.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "layout.cuh"
#include "ptx.cuh"

namespace sagefp4 {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& w, float (&v)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(u[i] << 16);
    v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// The rule of sage_fp4.h for one group, given its amax: returns the E4M3 byte
// and the reciprocal of the decoded scale (0 when the scale is 0).
__device__ __forceinline__ uint32_t group_scale(float amax, float& r) {
  const float q = __fdiv_rn(amax, 6.0f);
  const uint32_t sb = cvt_e4m3(q);
  const float s = e4m3_to_f32(sb);
  r = (s != 0.0f) ? __frcp_rn(s) : 0.0f;
  return sb;
}

__device__ __forceinline__ uint32_t encode8(const float (&v)[8], float r) {
  if (r == 0.0f) return 0u;
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(v[i], r);
  return cvt_e2m1x8(y);
}

// Q and K.  A row of D bf16 is D/8 lanes x 16 bytes; the two lanes holding one
// 16-element group combine their absmax with one shuffle.  Each warp keeps U
// row-steps of loads in flight.  blockIdx.y selects Q (0) or K (1).
template <int D>
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint4* __restrict__ x0,
                                                         const uint4* __restrict__ x1,
                                                         uint8_t* __restrict__ c0,
                                                         uint8_t* __restrict__ s0,
                                                         uint8_t* __restrict__ c1,
                                                         uint8_t* __restrict__ s1, int BH, int N,
                                                         int Np) {
  constexpr int LPR = D / 8;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp step
  constexpr int U = 4;
  const uint4* __restrict__ x = blockIdx.y ? x1 : x0;
  uint8_t* __restrict__ codes = blockIdx.y ? c1 : c0;
  uint8_t* __restrict__ scales = blockIdx.y ? s1 : s0;
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR;
  const int rsub = lane / LPR;
  const long long total = static_cast<long long>(BH) * Np / RPW;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;

  for (long long step0 = w0 * U; step0 < total; step0 += nwarps * U) {
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long row = (step0 + u) * RPW + rsub;
      const int bh = static_cast<int>(row / Np), n = static_cast<int>(row % Np);
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      if (step0 + u < total && n < N)
        raw[u] = __ldcs(x + (static_cast<size_t>(bh) * N + n) * (D / 8) + sub);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (step0 + u >= total) break;  // uniform across the warp
      const long long row = (step0 + u) * RPW + rsub;
      const int bh = static_cast<int>(row / Np), n = static_cast<int>(row % Np);
      float v[8];
      bf16x8_to_f32(raw[u], v);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
      float r;
      const uint32_t sb = group_scale(amax, r);
      const uint32_t word = encode8(v, r);
      *reinterpret_cast<uint32_t*>(codes + (static_cast<size_t>(bh) * Np + n) * (D / 2) +
                                   sub * 4) = word;
      // four consecutive groups' scales form one 32-bit word of the block layout
      const uint32_t w = sb | (__shfl_down_sync(kFull, sb, 2) << 8) |
                         (__shfl_down_sync(kFull, sb, 4) << 16) |
                         (__shfl_down_sync(kFull, sb, 6) << 24);
      if ((sub & 7) == 0) {
        const int g = sub / 2;
        *reinterpret_cast<uint32_t*>(scales + static_cast<size_t>(bh) * Np * (D / 16) +
                                     sf_offset(n, g, D / 16)) = w;
      }
    }
  }
}

// V.  One block stages 128 tokens x D channels in shared memory, then each
// thread quantizes a channel pair over 64 tokens (4 groups along tokens) and
// writes 32 contiguous code bytes per channel row of V^T plus one scale word.
template <int D>
__global__ void __launch_bounds__(128) quant_v_kernel(const uint4* __restrict__ v,
                                                      uint8_t* __restrict__ vc,
                                                      uint8_t* __restrict__ vs, int N, int Np) {
  __shared__ __align__(16) uint32_t tile[128 * (D / 2)];  // [token][channel pair] bf16x2
  const int ntiles = Np / 128;
  const int tb = static_cast<int>(blockIdx.x % ntiles);
  const int bh = static_cast<int>(blockIdx.x / ntiles);
  const int tid = threadIdx.x;
  constexpr int CH = D / 8;  // 16-byte chunks per token row
  for (int i = tid; i < 128 * CH; i += 128) {
    const int t = i / CH, c = i % CH;
    const int n = tb * 128 + t;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (n < N) val = __ldcs(v + (static_cast<size_t>(bh) * N + n) * CH + c);
    *reinterpret_cast<uint4*>(&tile[t * (D / 2) + c * 4]) = val;
  }
  __syncthreads();

  const size_t vt_row = static_cast<size_t>(Np) / 2;
  uint8_t* __restrict__ vs_bh = vs + static_cast<size_t>(bh) * 8 * Np;
  for (int it = tid; it < D; it += 128) {
    const int pch = it % (D / 2);  // channel pair
    const int h = it / (D / 2);    // 64-token half of the tile
    uint32_t clo[8], chi[8];
    uint32_t slo = 0, shi = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float lo[16], hi[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t w = tile[(h * 64 + g * 16 + j) * (D / 2) + pch];
        lo[j] = __uint_as_float(w << 16);
        hi[j] = __uint_as_float(w & 0xFFFF0000u);
      }
      float alo = 0.0f, ahi = 0.0f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        alo = fmaxf(alo, fabsf(lo[j]));
        ahi = fmaxf(ahi, fabsf(hi[j]));
      }
      float rlo, rhi;
      slo |= group_scale(alo, rlo) << (8 * g);
      shi |= group_scale(ahi, rhi) << (8 * g);
      float t8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) t8[j] = lo[j];
      clo[2 * g] = encode8(t8, rlo);
#pragma unroll
      for (int j = 0; j < 8; ++j) t8[j] = lo[8 + j];
      clo[2 * g + 1] = encode8(t8, rlo);
#pragma unroll
      for (int j = 0; j < 8; ++j) t8[j] = hi[j];
      chi[2 * g] = encode8(t8, rhi);
#pragma unroll
      for (int j = 0; j < 8; ++j) t8[j] = hi[8 + j];
      chi[2 * g + 1] = encode8(t8, rhi);
    }
    const int d0 = 2 * pch, d1 = 2 * pch + 1;
    uint8_t* row0 = vc + (static_cast<size_t>(bh) * D + d0) * vt_row + tb * 64 + h * 32;
    uint8_t* row1 = vc + (static_cast<size_t>(bh) * D + d1) * vt_row + tb * 64 + h * 32;
    reinterpret_cast<uint4*>(row0)[0] = make_uint4(clo[0], clo[1], clo[2], clo[3]);
    reinterpret_cast<uint4*>(row0)[1] = make_uint4(clo[4], clo[5], clo[6], clo[7]);
    reinterpret_cast<uint4*>(row1)[0] = make_uint4(chi[0], chi[1], chi[2], chi[3]);
    reinterpret_cast<uint4*>(row1)[1] = make_uint4(chi[4], chi[5], chi[6], chi[7]);
    const int g0 = tb * 8 + h * 4;
    *reinterpret_cast<uint32_t*>(vs_bh + sf_offset(d0, g0, Np / 16)) = slo;
    *reinterpret_cast<uint32_t*>(vs_bh + sf_offset(d1, g0, Np / 16)) = shi;
  }
  // scale rows of the padding channels D..127 of the 128-row block are zero
  for (int it = tid; it < (128 - D) * 2; it += 128) {
    const int d = D + it / 2, h = it % 2;
    *reinterpret_cast<uint32_t*>(vs_bh + sf_offset(d, tb * 8 + h * 4, Np / 16)) = 0u;
  }
}

int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

}  // namespace

cudaError_t launch_quant_rows(const void* q, const void* k, uint8_t* qc, uint8_t* qs, uint8_t* kc,
                              uint8_t* ks, int BH, int N, int D, cudaStream_t st) {
  const int Np = round_up_int(N, 128);
  const long long rows = static_cast<long long>(BH) * Np;
  const long long warps_needed = (rows * D / 256 + 3) / 4;  // a warp covers 256 elements per step, 4 steps
  long long blocks = (warps_needed + 7) / 8;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  dim3 grid(static_cast<unsigned>(blocks), 2);
  if (D == 128)
    quant_rows_kernel<128><<<grid, 256, 0, st>>>(static_cast<const uint4*>(q),
                                                 static_cast<const uint4*>(k), qc, qs, kc, ks, BH,
                                                 N, Np);
  else
    quant_rows_kernel<64><<<grid, 256, 0, st>>>(static_cast<const uint4*>(q),
                                                static_cast<const uint4*>(k), qc, qs, kc, ks, BH,
                                                N, Np);
  return cudaGetLastError();
}

cudaError_t launch_quant_v(const void* v, uint8_t* vc, uint8_t* vs, int BH, int N, int D,
                           cudaStream_t st) {
  const int Np = round_up_int(N, 128);
  const long long blocks = static_cast<long long>(Np / 128) * BH;
  const unsigned grid = static_cast<unsigned>(blocks);
  if (D == 128)
    quant_v_kernel<128><<<grid, 128, 0, st>>>(static_cast<const uint4*>(v), vc, vs, N, Np);
  else
    quant_v_kernel<64><<<grid, 128, 0, st>>>(static_cast<const uint4*>(v), vc, vs, N, Np);
  return cudaGetLastError();
}

}  // namespace sagefp4

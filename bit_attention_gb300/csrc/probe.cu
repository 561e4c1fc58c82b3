// probe.cu -- diagnostic kernels that expose the device primitives the
// attention path is built from, so that tests can pin them one at a time:
//   * the FP32 -> E2M1 / E4M3 conversions, over any range of bit patterns;
//   * one block-scaled FP4 tensor-core product of a 128-row tile, with its
//     operands staged exactly as the attention kernel stages Q/K/V (TMA with
//     hardware swizzle) or P (thread stores into the swizzled layout);
//   * the reducing tensor-memory load (values and their maximum per 16
//     columns) the attention kernel takes its group maxima from.
#include <cuda_fp16.h>

#include "../../include/sage_fp4.h"
#include "kernels.h"
#include "layout.cuh"
#include "ptx.cuh"

namespace sagefp4 {

namespace {

__global__ void cvt_probe_kernel(uint32_t first, uint32_t count, uint8_t* e2m1, uint8_t* e4m3) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += stride) {
    const float x = __uint_as_float(first + static_cast<uint32_t>(i));
    if (e2m1) e2m1[i] = static_cast<uint8_t>(cvt_e2m1x2(x, 0.0f));
    if (e4m3) e4m3[i] = static_cast<uint8_t>(cvt_e4m3(x));
  }
}

constexpr uint64_t kProbeWaitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ bool probe_wait(uint32_t bar, uint32_t parity, int32_t* err) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kProbeWaitNs) {
      atomicCAS(err, 0, SAGE_FP4_ETIMEOUT);
      return false;
    }
  }
  return true;
}

// Physical 16-byte chunk of logical chunk c in row r of a K-major tile with
// rows of RB bytes under the matching swizzle (32/64/128-byte).
template <int RB>
__device__ __forceinline__ int swz_chunk(int r, int c) {
  if (RB == 32) return c ^ ((r >> 2) & 1);
  if (RB == 64) return c ^ ((r >> 1) & 3);
  return c ^ (r & 7);
}

template <int K>
__global__ void __launch_bounds__(128, 1)
    mma_probe_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                     const MmaProbeParams p, int32_t* err) {
  constexpr int RB = K / 2;          // bytes per operand row
  constexpr int KB = K / 64;         // MMAs (K = 64 each)
  constexpr uint32_t swz = (RB == 32) ? kSwizzle32B : (RB == 64) ? kSwizzle64B : kSwizzle128B;
  constexpr uint32_t sbo = 8 * RB;
  // each operand's scales: KB * 512 bytes (block layout) at the start of a
  // 48 KB region; in the 128-row mode, step kb's 128-row copy source at
  // 4096 + 2048 kb, and noise everywhere else (the region covers every read of
  // the 128-row copies under either reading of the descriptor's two strides)
  constexpr int kSfRegion = 49152, kSfRows = 4096;
  constexpr int oA = 0, oB = 128 * RB, oSFA = 2 * 128 * RB, oSFB = oSFA + kSfRegion,
                oBar = oSFB + kSfRegion, oSlot = oBar + 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int warp = threadIdx.x >> 5;
  const uint32_t bar_load = sb + oBar, bar_mma = sb + oBar + 8;
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + oSlot);

  if (threadIdx.x == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (threadIdx.x == 0) {
    const uint32_t bytes = (p.a_by_threads ? 0 : 128 * RB) + p.n * RB + 2 * KB * 512;
    mbar_arrive_expect_tx(bar_load, bytes);
    if (!p.a_by_threads) tma_load_2d(sb + oA, &ta, 0, 0, bar_load);
    tma_load_2d(sb + oB, &tb, 0, 0, bar_load);
    bulk_load(sb + oSFA, p.a_scales, KB * 512, bar_load);
    bulk_load(sb + oSFB, p.b_scales, KB * 512, bar_load);
  }
  // noise after the scales: every value, NaN encodings included (E4M3 0x7F,
  // E8M0 0xFF), so that a product that read it would show
  for (int i = KB * 512 + static_cast<int>(threadIdx.x); i < kSfRegion; i += blockDim.x) {
    const uint8_t v = (i % 5 == 0) ? 0x7F : (i % 7 == 0) ? 0xFF : static_cast<uint8_t>(i * 37 + 11);
    sm[oSFA + i] = v;
    sm[oSFB + i] = static_cast<uint8_t>(v ^ 0x80);
  }
  __syncthreads();
  if (p.sf_rows128) {
    // A's 128-row copy source of step kb: row r (16 bytes) holds, in its word
    // r / 32, the scale word of matrix row r (the block layout keeps it at row
    // r % 32, word r / 32); its other three words stay noise
    for (int i = threadIdx.x; i < KB * 128; i += blockDim.x) {
      const int kb = i / 128, r = i % 128;
      const int src = 512 * kb + (r % 32) * 16 + (r / 32) * 4;
      const int dst = kSfRows + 2048 * kb + r * 16 + (r / 32) * 4;
      *reinterpret_cast<uint32_t*>(sm + oSFA + dst) = *reinterpret_cast<const uint32_t*>(p.a_scales + src);
    }
  }
  fence_proxy_async_smem();
  if (p.a_by_threads) {
    for (int i = threadIdx.x; i < 128 * (RB / 16); i += blockDim.x) {
      const int r = i / (RB / 16), c = i % (RB / 16);
      const uint4 v = reinterpret_cast<const uint4*>(p.a_codes + r * RB)[c];
      *reinterpret_cast<uint4*>(sm + oA + r * RB + swz_chunk<RB>(r, c) * 16) = v;
    }
    fence_proxy_async_smem();
  }
  __syncthreads();

  bool ok = true;
  if (threadIdx.x == 0) {
    ok = probe_wait(bar_load, 0, err);
    if (ok) {
      tc_fence_after();
      // B's scales: every lane quarter holds all rows (each quarter of the
      // MMA's output rows reads them from its own quarter)
      for (int kb = 0; kb < KB; ++kb)
        tc_cp_32x128b_warpx4(tmem + 160 + 4 * kb, smem_desc(sb + oSFB + 512 * kb, 0, 128, kSwizzleNone));
      if (!p.sf_rows128) {
        for (int kb = 0; kb < KB; ++kb)
          tc_cp_32x128b_warpx4(tmem + 128 + 4 * kb, smem_desc(sb + oSFA + 512 * kb, 0, 128, kSwizzleNone));
      } else if (KB == 1) {
        tc_cp_128x128b(tmem + 128, smem_desc(sb + oSFA + kSfRows, 0, 128, kSwizzleNone));
      } else {
        // two steps per copy: the second 16 bytes of row r are step 2j+1's row r
        for (int j = 0; j < KB / 2; ++j)
          tc_cp_128x256b(tmem + 128 + 8 * j, smem_desc(sb + oSFA + kSfRows + 4096 * j, 2048, 128, kSwizzleNone));
      }
      const uint32_t n = static_cast<uint32_t>(p.n);
      for (int kb = 0; kb < KB; ++kb) {
        const uint64_t ad = smem_desc(sb + oA + 32 * kb, 16, sbo, swz);
        const uint64_t bd = smem_desc(sb + oB + 32 * kb, 16, sbo, swz);
        if (p.mx)
          mma_mxf4(tmem, ad, bd, idesc_mxf4(128, n), tmem + 128 + 4 * kb, tmem + 160 + 4 * kb, kb > 0);
        else
          mma_nvfp4(tmem, ad, bd, idesc_nvfp4(128, n), tmem + 128 + 4 * kb, tmem + 160 + 4 * kb, kb > 0);
      }
      tc_commit(bar_mma);
    }
  }
  __syncthreads();
  ok = (*reinterpret_cast<volatile int32_t*>(err) == 0);
  if (ok && probe_wait(bar_mma, 0, err)) {
    tc_fence_after();
    const int r = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    for (int c = 0; c < p.n / 16; ++c) {
      uint32_t v[16];
      tmem_ld16(tmem + c * 16 + lane_base, v);
      tmem_wait_ld();
      for (int i = 0; i < 16; ++i) p.d[r * p.n + c * 16 + i] = __uint_as_float(v[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int K>
cudaError_t launch_mma_probe_k(const CUtensorMap& ta, const CUtensorMap& tb,
                               const MmaProbeParams& p, cudaStream_t st) {
  const int smem = 2 * 128 * (K / 2) + 2 * 49152 + 64 + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(mma_probe_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mma_probe_kernel<K><<<1, 128, smem, st>>>(ta, tb, p, p.status);
  return cudaGetLastError();
}

// Tensor-core rate of the attention kernel's MMA instruction: one CTA per
// SM, one thread issuing `iters` back-to-back block-scaled FP4 MMAs (D += A
// B^T, M = 128, N = n, K = 64) on operands held in shared memory (bytes of
// a fixed pseudo-random pattern), then one commit.  The caller times the
// launch; FLOPs = 2 * 128 * n * 64 * iters per CTA.
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int n, int32_t* err) {
  constexpr int oA = 0, oB = 4096, oSF = oB + 256 * 32, oBar = oSF + 3 * 512;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int warp = threadIdx.x >> 5;
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + oBar + 8);
  // operand bytes: a fixed pattern; scale bytes: E4M3 values 0.5 .. 2
  for (int i = threadIdx.x; i < oSF / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sm)[i] = (static_cast<uint32_t>(i) * 2654435761u) ^ 0x5A5A5A5Au;
  for (int i = threadIdx.x; i < 3 * 512; i += blockDim.x) sm[oSF + i] = static_cast<uint8_t>(0x30 + (i * 7) % 16);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(sb + oBar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (threadIdx.x == 0) {
    // scale factors: A in columns 256..259, B in 264..271 (two 128-row blocks)
    tc_cp_32x128b_warpx4(tmem + 256, smem_desc(sb + oSF, 0, 128, kSwizzleNone));
    tc_cp_32x128b_warpx4(tmem + 264, smem_desc(sb + oSF + 512, 0, 128, kSwizzleNone));
    tc_cp_32x128b_warpx4(tmem + 268, smem_desc(sb + oSF + 1024, 0, 128, kSwizzleNone));
    const uint64_t ad = smem_desc(sb + oA, 16, 8 * 32, kSwizzle32B);
    const uint64_t bd = smem_desc(sb + oB, 16, 8 * 32, kSwizzle32B);
    const uint32_t idesc = idesc_nvfp4(128, static_cast<uint32_t>(n));
    for (int i = 0; i < iters; ++i) mma_nvfp4(tmem, ad, bd, idesc, tmem + 256, tmem + 264, i > 0);
    tc_commit(sb + oBar);
    probe_wait(sb + oBar, 0, err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The reducing tensor-memory load the attention kernel uses for group
// maxima: one CTA of 128 threads stores in[r][0..127] (FP32, row r = lane r)
// into 128 tensor-memory columns, reads them back in eight 16-column groups
// with tcgen05.ld.red ... max, and writes the values it got to vals[r][..]
// and the reported maxima to maxes[r][0..7].
__global__ void __launch_bounds__(128, 1)
    tmem_max_probe_kernel(const float* __restrict__ in, float* __restrict__ vals, float* __restrict__ maxes) {
  __shared__ uint32_t slot;
  const int warp = threadIdx.x >> 5, r = threadIdx.x;
  if (warp == 0) {
    tmem_alloc(smem_addr(&slot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tb = slot + lane_base;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __float_as_uint(in[r * 128 + 8 * c + j]);
    tmem_st8(tb + 8 * c, w);
  }
  tmem_wait_st();
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    uint32_t v[16];
    float mx;
    tmem_ld16_max(tb + 16 * g, v, mx);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) vals[r * 128 + 16 * g + j] = __uint_as_float(v[j]);
    maxes[r * 8 + g] = mx;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(slot, 128);
  }
}

}  // namespace

cudaError_t launch_tmem_max_probe(const float* in, float* vals, float* maxes, cudaStream_t st) {
  tmem_max_probe_kernel<<<1, 128, 0, st>>>(in, vals, maxes);
  return cudaGetLastError();
}

cudaError_t launch_cvt_probe(uint32_t first, uint32_t count, uint8_t* e2m1, uint8_t* e4m3,
                             cudaStream_t st) {
  unsigned blocks = (count + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (blocks == 0) blocks = 1;
  cvt_probe_kernel<<<blocks, 256, 0, st>>>(first, count, e2m1, e4m3);
  return cudaGetLastError();
}

cudaError_t launch_mma_peak(int iters, int n, int32_t* status, cudaStream_t st) {
  const int smem = 4096 + 256 * 32 + 3 * 512 + 64 + 1024;
  cudaError_t e = cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  mma_peak_kernel<<<sms > 0 ? sms : 1, 128, smem, st>>>(iters, n, status);
  return cudaGetLastError();
}

cudaError_t launch_mma_probe(const CUtensorMap& ta, const CUtensorMap& tb, const MmaProbeParams& p,
                             cudaStream_t st) {
  if (p.K == 64) return launch_mma_probe_k<64>(ta, tb, p, st);
  if (p.K == 128) return launch_mma_probe_k<128>(ta, tb, p, st);
  return launch_mma_probe_k<256>(ta, tb, p, st);
}

}  // namespace sagefp4

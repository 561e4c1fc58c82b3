// quant.cu -- NVFP4 quantization of Q, K (groups of 16 along D) and V (groups
// of 16 along tokens, written as V^T), bit-exact with the rule in sage_fp4.h;
// and the MXFP4 variant (groups of 32, E8M0 scales, same layouts).
//
// Method: 1x16 microscaling of both products (senqingzn.com article on
// SageAttention3, "Solving two obstacles and one difficulty", solution 1);
// NVFP4 = E2M1 codes + one E4M3 scale per 16 elements ("FP4 attention
// inference acceleration and hardware implementation/optimisation").
//
// Both kernels are HBM-bound streams: 2 bytes read and 0.5625 bytes written
// per element.  The per-group arithmetic is kept short: amax/6 is one
// multiply with an FMA residual correction (equal to the correctly rounded
// quotient for every bf16 amax), and 1/scale comes from a 256-entry table of
// correctly rounded reciprocals of the E4M3 values.
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

// Round-to-nearest amax / 6 for amax a bf16 magnitude: q0 = amax * RN(1/6),
// then one FMA-computed residual step.  Checked against correctly rounded
// division for all 32640 non-negative finite bf16 values.
__device__ __forceinline__ float div6(float amax) {
  const float y = 0.16666667163372040f;  // RN(1/6)
  const float q0 = __fmul_rn(amax, y);
  const float r = __fmaf_rn(-6.0f, q0, amax);
  return __fmaf_rn(r, y, q0);
}

// rtab[b] = RN(1 / value(E4M3 byte b)) for positive finite b, 0 otherwise.
__device__ __forceinline__ void fill_rtab(float* rtab) {
  for (int b = threadIdx.x; b < 256; b += blockDim.x) {
    const float s = e4m3_to_f32(static_cast<uint32_t>(b));
    rtab[b] = (b > 0 && b < 0x7F) ? __frcp_rn(s) : 0.0f;
  }
}

// Eight values times the group's reciprocal scale, then E2M1.  The products
// are taken two at a time (mul.rn.f32x2: each lane rounded like __fmul_rn).
__device__ __forceinline__ uint32_t encode8(const float (&v)[8], float r) {
  const uint64_t rr = pack2(r, r);
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const uint64_t p = mul2(pack2(v[i], v[i + 1]), rr);
    y[i] = lo2(p);
    y[i + 1] = hi2(p);
  }
  return cvt_e2m1x8(y);
}

// Lane-wise max(|a|, |b|) of two packed bf16 pairs; the sign bit of each
// result is the XOR of the operands' signs and is discarded by the caller.
// Exact for finite inputs.
__device__ __forceinline__ uint32_t maxabs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Bytes b0..b3 (each in bits 0-7 of its argument) packed into one word.
__device__ __forceinline__ uint32_t pack4_bytes(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// Q and K.  A row of D bf16 is D/8 lanes x 16 bytes; the two lanes holding one
// 16-element group combine their absmax with one shuffle.  A warp handles a
// chunk of 8 row-steps (16 rows for D = 128, 32 for D = 64) of one (b,h);
// chunks never straddle two heads because N_pad is a multiple of 128, and lie
// inside one 32-row slice of the scale block layout, so a lane's scale address
// moves by a constant from one row-step to the next.  The warp keeps all its
// row-steps' loads in flight before it computes.  blockIdx.y selects Q (0) or
// K (1); each input has its own strides (elements, multiples of 8).  MX: a
// group of 32 spans four lanes, and each K = 64 step's scale word holds the
// two E8M0 bytes in its low half.
template <int D, bool MX>
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint4* __restrict__ x0,
                                                         const uint4* __restrict__ x1,
                                                         Strides t0, Strides t1,
                                                         uint8_t* __restrict__ c0,
                                                         uint8_t* __restrict__ s0,
                                                         uint8_t* __restrict__ c1,
                                                         uint8_t* __restrict__ s1, int H, int BH,
                                                         int N, int Np, const Extents ext) {
  constexpr int LPR = D / 8;      // lanes per row
  constexpr int RPW = 32 / LPR;   // rows per warp step
  constexpr int U = 8;            // row-steps per chunk
  constexpr int CHUNK = U * RPW;  // rows per warp chunk
  static_assert(32 % CHUNK == 0, "a chunk must sit inside one 32-row slice");
  __shared__ float rtab[256];
  fill_rtab(rtab);
  __syncthreads();
  // the V kernel queued after this grid may start now (it touches other memory)
  griddep_launch_dependents();
  const uint4* __restrict__ x = blockIdx.y ? x1 : x0;
  const Strides t = blockIdx.y ? t1 : t0;
  const size_t step = static_cast<size_t>(RPW) * static_cast<size_t>(t.n / 8);  // one row-step, in uint4
  uint8_t* __restrict__ codes = blockIdx.y ? c1 : c0;
  uint8_t* __restrict__ scales = blockIdx.y ? s1 : s0;
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR;
  const int rsub = lane / LPR;
  const int chunks_per_head = Np / CHUNK;
  const int total = BH * chunks_per_head;  // BH * Np <= INT_MAX is checked on the host
  const int nwarps = static_cast<int>((gridDim.x * blockDim.x) >> 5);
  for (int chunk = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5); chunk < total;
       chunk += nwarps) {
    const int bh = chunk / chunks_per_head;
    const int r0 = (chunk - bh * chunks_per_head) * CHUNK;
    const int n0 = r0 + rsub;
    const int b = bh / H, h = bh - b * H;
    const long long off0 = b * t.b + h * t.h + static_cast<long long>(n0) * t.n + sub * 8;  // elements
    const uint4* __restrict__ src = x + static_cast<size_t>(off0 / 8);
    const long long xext = ext.x[blockIdx.y];
    uint4 raw[U];
    if (r0 + CHUNK <= N) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        raw[u] = in_bounds(ext, off0 + u * RPW * t.n, 8, xext) ? __ldcs(src + u * step)
                                                               : make_uint4(0u, 0u, 0u, 0u);
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u)
        raw[u] = (n0 + u * RPW < N && in_bounds(ext, off0 + u * RPW * t.n, 8, xext)) ? __ldcs(src + u * step)
                                                                                     : make_uint4(0u, 0u, 0u, 0u);
    }
    uint8_t* __restrict__ cdst = codes + (static_cast<size_t>(bh) * Np + n0) * (D / 2) + sub * 4;
    uint8_t* __restrict__ sdst =
        scales + static_cast<size_t>(bh) * Np * (D / 16) + sf_offset(n0, sub / 2, D / 16);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint4 w = raw[u];
      uint32_t m = maxabs_bf16x2(maxabs_bf16x2(w.x, w.y), maxabs_bf16x2(w.z, w.w));
      m = maxabs_bf16x2(m, __shfl_xor_sync(kFull, m, 1));
      if constexpr (MX) m = maxabs_bf16x2(m, __shfl_xor_sync(kFull, m, 2));
      const float amax = fmaxf(fabsf(__uint_as_float(m << 16)), fabsf(__uint_as_float(m & 0xFFFF0000u)));
      float v[8];
      bf16x8_to_f32(w, v);
      uint32_t word, sw;
      if constexpr (MX) {
        const uint32_t e8 = e8m0_of(amax);
        word = encode8(v, e8m0_mult(e8));
        sw = pack4_bytes(e8, __shfl_down_sync(kFull, e8, 4), 0u, 0u);
      } else {
        const uint32_t sb = cvt_e4m3(div6(amax));
        const float r = rtab[sb];
        word = (r != 0.0f) ? encode8(v, r) : 0u;
        // four consecutive groups' scales form one 32-bit word of the block layout
        sw = pack4_bytes(sb, __shfl_down_sync(kFull, sb, 2), __shfl_down_sync(kFull, sb, 4),
                         __shfl_down_sync(kFull, sb, 6));
      }
      if (in_bounds(ext, (cdst + u * RPW * (D / 2)) - codes, 4, ext.codes))
        *reinterpret_cast<uint32_t*>(cdst + u * RPW * (D / 2)) = word;
      if ((sub & 7) == 0 && in_bounds(ext, (sdst + u * RPW * 16) - scales, 4, ext.scales))
        *reinterpret_cast<uint32_t*>(sdst + u * RPW * 16) = sw;
    }
  }
}

// V.  Each block walks TT-token tiles of V (tile i of this block = blockIdx.x
// + i * gridDim.x over (b,h) x tiles).  A tile is brought into shared memory
// as [TT tokens][D channels] by bulk copies into an NS-deep ring, so that the
// next NS-1 tiles load while this one is quantized: one copy of the whole
// tile when a head's tokens are contiguous (token stride D), else one copy
// per token row, spread over the lanes of warp 0.  A work item is one channel
// pair over 32 tokens (two groups along tokens): it writes 16 code bytes to
// each of two V^T rows and one 16-bit half of a scale word per row.  MX: the
// 32 tokens are one group; its E8M0 byte goes to byte `seg` of the tile's
// scale word (a 64-token tile is one K = 64 step), and seg 0 zeroes the
// word's upper half.
// Every wait for a tile is bounded by wait_ns; a wait that gives up sets
// *status to SAGE_FP4_ETIMEOUT and the whole block leaves together (one vote
// of all its threads decides), after the copies it still has in flight have
// landed.  withhold (failure-detection test only): block 0 never issues its
// first tile, so its wait for that tile runs out.
template <int D, int TT, int NS, bool MX>
__global__ void __launch_bounds__(128) quant_v_kernel(const uint8_t* __restrict__ v, Strides sv,
                                                      uint8_t* __restrict__ vc,
                                                      uint8_t* __restrict__ vs, int H, int BH,
                                                      int N, int Np, int32_t* status, uint64_t wait_ns,
                                                      int withhold, const Extents ext) {
  static_assert(TT == 64 || TT == 128, "tile of 64 or 128 tokens");
  static_assert(!MX || TT == 64, "MX scale words follow 64-token tiles");
  constexpr int TILE_BYTES = TT * D * 2;
  constexpr int ITEMS = (D / 2) * (TT / 32);
  extern __shared__ __align__(128) uint8_t qv_smem[];
  uint32_t* tiles = reinterpret_cast<uint32_t*>(qv_smem);  // NS x [TT tokens][D/2 pairs]
  __shared__ float rtab[256];
  __shared__ __align__(8) uint64_t bars[NS];
  fill_rtab(rtab);
  const int ntiles = Np / TT;
  const long long work = static_cast<long long>(BH) * ntiles;
  const uint32_t bar0 = smem_addr(&bars[0]);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(bar0 + 8 * i, 1);
    mbar_fence_init();
  }
  __syncthreads();

  // Token rows of tile w that hold data (those past N are not read; they are
  // zeroed).  With TT = 64 a tile can lie wholly in the padding.
  auto tile_rows = [&](long long w) -> int {
    const int tb = static_cast<int>(w % ntiles);
    return max(0, min(TT, N - tb * TT));
  };
  // Called by all of warp 0.  Lane 0 announces the bytes before any copy is
  // issued, so the phase cannot complete before every copy has landed.
  const int lane = threadIdx.x & 31;
  auto issue = [&](long long w, int buf) {
    const int bh = static_cast<int>(w / ntiles), tb = static_cast<int>(w % ntiles);
    const int b = bh / H, h = bh - b * H;
    const int rows = tile_rows(w);
    const long long off = b * sv.b + h * sv.h + static_cast<long long>(tb) * TT * sv.n;  // elements
    const uint8_t* src = v + off * 2;
    const uint32_t dst = smem_addr(qv_smem + buf * TILE_BYTES);
    if (lane == 0) mbar_arrive_expect_tx(bar0 + 8 * buf, static_cast<uint32_t>(rows) * D * 2);
    __syncwarp();
    // (debug build: a copy that would leave V is skipped; its tile's wait then
    // runs out, after the bounds failure has been recorded)
    if (sv.n == D) {
      if (lane == 0 && rows > 0 && in_bounds(ext, off, static_cast<long long>(rows) * D, ext.x[2]))
        bulk_load(dst, src, static_cast<uint32_t>(rows) * D * 2, bar0 + 8 * buf);
    } else {
      for (int r = lane; r < rows; r += 32)
        if (in_bounds(ext, off + static_cast<long long>(r) * sv.n, D, ext.x[2]))
          bulk_load(dst + r * D * 2, src + static_cast<long long>(r) * sv.n * 2, D * 2, bar0 + 8 * buf);
    }
  };
  if (threadIdx.x < 32)
    for (int s = 0; s < NS - 1; ++s) {
      const long long ws = blockIdx.x + static_cast<long long>(s) * gridDim.x;
      if (ws < work && !(withhold && blockIdx.x == 0 && s == 0)) issue(ws, s);
    }
  const size_t vt_row = static_cast<size_t>(Np) / 2;
  long long w = blockIdx.x;
  for (int it = 0; w < work; ++it, w += gridDim.x) {
    const int buf = it % NS;
    // refill the slot that the last iteration released at its closing barrier
    const long long wn = w + static_cast<long long>(NS - 1) * gridDim.x;
    if (threadIdx.x < 32 && wn < work) issue(wn, (it + NS - 1) % NS);
    // wait for this tile: every thread's wait is bounded
    bool ok = true;
    {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar0 + 8 * buf, (it / NS) & 1)) {
        if (globaltimer_ns() - t0 > wait_ns) {
          ok = false;
          break;
        }
      }
    }
    const int bh = static_cast<int>(w / ntiles), tb = static_cast<int>(w % ntiles);
    uint32_t* tile = tiles + buf * (TILE_BYTES / 4);
    const int rows = tile_rows(w);
    if (ok)
      for (int i = rows * (D / 2) + threadIdx.x; i < TT * (D / 2); i += 128) tile[i] = 0u;
    // one vote of the whole block (it also publishes the zeroed rows): if any
    // thread's wait gave up, every thread leaves
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        atomicCAS(status, 0, -3);  // SAGE_FP4_ETIMEOUT
        // let the copies already issued into the other slots land before exiting
        const uint64_t t1 = globaltimer_ns();
        for (int s = 1; s < NS; ++s) {
          const long long ws = w + static_cast<long long>(s) * gridDim.x;
          if (ws >= work) break;
          const int j = it + s;
          while (!mbar_try_wait(bar0 + 8 * (j % NS), (j / NS) & 1) && globaltimer_ns() - t1 < wait_ns) {
          }
        }
      }
      griddep_wait();
      return;
    }

    uint8_t* __restrict__ vs_bh = vs + static_cast<size_t>(bh) * 8 * Np;
    for (int item = threadIdx.x; item < ITEMS; item += 128) {
      const int pch = item % (D / 2);  // channel pair
      const int seg = item / (D / 2);  // 32-token segment of the tile
      if constexpr (MX) {
        uint32_t m = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) m = maxabs_bf16x2(m, tile[(seg * 32 + j) * (D / 2) + pch]);
        const uint32_t elo = e8m0_of(fabsf(__uint_as_float(m << 16)));
        const uint32_t ehi = e8m0_of(fabsf(__uint_as_float(m & 0xFFFF0000u)));
        const float rlo = e8m0_mult(elo), rhi = e8m0_mult(ehi);
        uint32_t clo[4], chi[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float lo[8], hi[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t wv = tile[(seg * 32 + q * 8 + j) * (D / 2) + pch];
            lo[j] = __uint_as_float(wv << 16);
            hi[j] = __uint_as_float(wv & 0xFFFF0000u);
          }
          clo[q] = encode8(lo, rlo);
          chi[q] = encode8(hi, rhi);
        }
        const int d0 = 2 * pch, d1 = 2 * pch + 1;
        const size_t col = static_cast<size_t>(tb) * (TT / 2) + seg * 16;
        const long long c0 = (static_cast<long long>(bh) * D + d0) * vt_row + col;
        const long long c1 = (static_cast<long long>(bh) * D + d1) * vt_row + col;
        const long long sbase = static_cast<long long>(bh) * 8 * Np;
        if (in_bounds(ext, c0, 16, ext.vt_codes))
          *reinterpret_cast<uint4*>(vc + c0) = make_uint4(clo[0], clo[1], clo[2], clo[3]);
        if (in_bounds(ext, c1, 16, ext.vt_codes))
          *reinterpret_cast<uint4*>(vc + c1) = make_uint4(chi[0], chi[1], chi[2], chi[3]);
        if (in_bounds(ext, sbase + sf_offset(d0, tb * 4 + seg, Np / 16), 1, ext.vt_scales))
          vs_bh[sf_offset(d0, tb * 4 + seg, Np / 16)] = static_cast<uint8_t>(elo);
        if (in_bounds(ext, sbase + sf_offset(d1, tb * 4 + seg, Np / 16), 1, ext.vt_scales))
          vs_bh[sf_offset(d1, tb * 4 + seg, Np / 16)] = static_cast<uint8_t>(ehi);
        if (seg == 0) {
          if (in_bounds(ext, sbase + sf_offset(d0, tb * 4 + 2, Np / 16), 2, ext.vt_scales))
            *reinterpret_cast<uint16_t*>(vs_bh + sf_offset(d0, tb * 4 + 2, Np / 16)) = 0;
          if (in_bounds(ext, sbase + sf_offset(d1, tb * 4 + 2, Np / 16), 2, ext.vt_scales))
            *reinterpret_cast<uint16_t*>(vs_bh + sf_offset(d1, tb * 4 + 2, Np / 16)) = 0;
        }
        continue;
      }
      uint32_t clo[4], chi[4];
      uint32_t sbl[2], sbh[2];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        float lo[16], hi[16];
        uint32_t m = 0u;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t wv = tile[(seg * 32 + g * 16 + j) * (D / 2) + pch];
          m = maxabs_bf16x2(m, wv);  // both channels' running absmax at once
          lo[j] = __uint_as_float(wv << 16);
          hi[j] = __uint_as_float(wv & 0xFFFF0000u);
        }
        const float alo = fabsf(__uint_as_float(m << 16));
        const float ahi = fabsf(__uint_as_float(m & 0xFFFF0000u));
        sbl[g] = cvt_e4m3(div6(alo));
        sbh[g] = cvt_e4m3(div6(ahi));
        const float rlo = rtab[sbl[g]], rhi = rtab[sbh[g]];
        float t8[8];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
#pragma unroll
          for (int j = 0; j < 8; ++j) t8[j] = lo[8 * q + j];
          clo[2 * g + q] = (rlo != 0.0f) ? encode8(t8, rlo) : 0u;
#pragma unroll
          for (int j = 0; j < 8; ++j) t8[j] = hi[8 * q + j];
          chi[2 * g + q] = (rhi != 0.0f) ? encode8(t8, rhi) : 0u;
        }
      }
      const int d0 = 2 * pch, d1 = 2 * pch + 1;
      const size_t col = static_cast<size_t>(tb) * (TT / 2) + seg * 16;
      const long long c0 = (static_cast<long long>(bh) * D + d0) * vt_row + col;
      const long long c1 = (static_cast<long long>(bh) * D + d1) * vt_row + col;
      const long long sbase = static_cast<long long>(bh) * 8 * Np;
      if (in_bounds(ext, c0, 16, ext.vt_codes))
        *reinterpret_cast<uint4*>(vc + c0) = make_uint4(clo[0], clo[1], clo[2], clo[3]);
      if (in_bounds(ext, c1, 16, ext.vt_codes))
        *reinterpret_cast<uint4*>(vc + c1) = make_uint4(chi[0], chi[1], chi[2], chi[3]);
      const int g0 = tb * (TT / 16) + seg * 2;  // even: the two groups share a 16-bit half
      if (in_bounds(ext, sbase + sf_offset(d0, g0, Np / 16), 2, ext.vt_scales))
        *reinterpret_cast<uint16_t*>(vs_bh + sf_offset(d0, g0, Np / 16)) =
            static_cast<uint16_t>(sbl[0] | (sbl[1] << 8));
      if (in_bounds(ext, sbase + sf_offset(d1, g0, Np / 16), 2, ext.vt_scales))
        *reinterpret_cast<uint16_t*>(vs_bh + sf_offset(d1, g0, Np / 16)) =
            static_cast<uint16_t>(sbh[0] | (sbh[1] << 8));
    }
    // scale rows of the padding channels D..127 of the 128-row block are zero
    for (int i = threadIdx.x; i < (128 - D) * (TT / 64); i += 128) {
      const int d = D + i / (TT / 64), h = i % (TT / 64);
      if (in_bounds(ext, static_cast<long long>(bh) * 8 * Np + sf_offset(d, tb * (TT / 16) + h * 4, Np / 16), 4,
                    ext.vt_scales))
        *reinterpret_cast<uint32_t*>(vs_bh + sf_offset(d, tb * (TT / 16) + h * 4, Np / 16)) = 0u;
    }
    // this slot is refilled by a bulk copy (async proxy) after the barrier
    fence_proxy_async_smem();
    __syncthreads();
  }
  // This grid may have started while the Q and K grid before it was still
  // running; it ends only after that grid, so work queued after it sees both.
  griddep_wait();
}

int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

}  // namespace

cudaError_t launch_quant_rows(const void* q, const void* k, Strides sq, Strides sk, uint8_t* qc,
                              uint8_t* qs, uint8_t* kc, uint8_t* ks, int H, int BH, int N, int D,
                              bool mx, const Extents& ext, cudaStream_t st) {
  const int Np = round_up_int(N, 128);
  const long long chunks = static_cast<long long>(BH) * Np / (D == 128 ? 16 : 32);  // one warp each
  long long blocks = (chunks + 7) / 8;
  // D = 128: one wave of 8 resident blocks per SM (4 per tensor), so that the
  // V grid queued behind may start at once (measured on GB300: +3% on the LLM
  // shape over two waves); D = 64: 8 per tensor (two waves), measured best
  const long long cap = static_cast<long long>(num_sms()) * (D == 128 ? 4 : 8);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  dim3 grid(static_cast<unsigned>(blocks), 2);
  const uint4* x0 = static_cast<const uint4*>(q);
  const uint4* x1 = static_cast<const uint4*>(k);
  if (D == 128) {
    if (mx)
      quant_rows_kernel<128, true><<<grid, 256, 0, st>>>(x0, x1, sq, sk, qc, qs, kc, ks, H, BH, N, Np, ext);
    else
      quant_rows_kernel<128, false><<<grid, 256, 0, st>>>(x0, x1, sq, sk, qc, qs, kc, ks, H, BH, N, Np, ext);
  } else {
    if (mx)
      quant_rows_kernel<64, true><<<grid, 256, 0, st>>>(x0, x1, sq, sk, qc, qs, kc, ks, H, BH, N, Np, ext);
    else
      quant_rows_kernel<64, false><<<grid, 256, 0, st>>>(x0, x1, sq, sk, qc, qs, kc, ks, H, BH, N, Np, ext);
  }
  return cudaGetLastError();
}

template <int D, int TT, int NS, bool MX>
cudaError_t launch_quant_v_cfg(const void* v, Strides sv, uint8_t* vc, uint8_t* vs, int H, int BH,
                               int Np, int N, int32_t* status, int blocks_per_sm, uint64_t wait_ns,
                               int withhold, const Extents& ext, cudaStream_t st) {
  const long long work = static_cast<long long>(Np / TT) * BH;
  const int smem = NS * TT * D * 2;
  long long blocks = static_cast<long long>(num_sms()) * blocks_per_sm;
  if (blocks > work) blocks = work;
  if (blocks < 1) blocks = 1;
  const cudaError_t e = cudaFuncSetAttribute(quant_v_kernel<D, TT, NS, MX>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the grid may start while the Q and K grid
  // queued before it drains (they touch disjoint memory; every block of that
  // grid is already running by then, so this grid's waiting blocks cannot
  // hold it back).  Measured: quantization 3-4% faster, bit-identical.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_v_kernel<D, TT, NS, MX>, static_cast<const uint8_t*>(v), sv, vc, vs,
                            H, BH, N, Np, status, wait_ns, withhold, ext);
}

cudaError_t launch_quant_v(const void* v, Strides sv, uint8_t* vc, uint8_t* vs, int H, int BH, int N,
                           int D, bool mx, int32_t* status, uint64_t wait_ns, int withhold,
                           const Extents& ext, cudaStream_t st) {
  const int Np = round_up_int(N, 128);
  // 64-token tiles, double-buffered: 32 KB (D = 128) or 16 KB (D = 64) of
  // shared memory per block.  The per-tile arithmetic, not the copy latency,
  // sets the pace, so several resident blocks beat deeper rings (measured on
  // GB300: 5.3-5.8 TB/s at D = 128 with six blocks per SM, against 4.0-4.9 TB/s
  // with four-deep rings and two or three blocks).  Five blocks per SM at
  // D = 128 leave room for the Q/K grid's last blocks: 1-3% faster than six
  // on every D = 128 workload.
  if (D == 128)
    return mx ? launch_quant_v_cfg<128, 64, 2, true>(v, sv, vc, vs, H, BH, Np, N, status, 5, wait_ns, withhold, ext, st)
              : launch_quant_v_cfg<128, 64, 2, false>(v, sv, vc, vs, H, BH, Np, N, status, 5, wait_ns, withhold, ext, st);
  return mx ? launch_quant_v_cfg<64, 64, 2, true>(v, sv, vc, vs, H, BH, Np, N, status, 8, wait_ns, withhold, ext, st)
            : launch_quant_v_cfg<64, 64, 2, false>(v, sv, vc, vs, H, BH, Np, N, status, 8, wait_ns, withhold, ext, st);
}

}  // namespace sagefp4

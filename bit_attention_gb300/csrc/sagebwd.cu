// sagebwd.cu -- SageBwd, the 8-bit attention for training: forward and
// backward kernels and the C ABI of include/sagebwd.h (senqingzn.com article
// on SageAttention3, "INT8 attention for training" and "Solving two obstacles
// and one difficulty", difficulty 3; abstract of "SageAttention3: Microscaling
// FP4 Attention for Inference and An Exploration of 8-Bit Training").
//
// Six of the seven products take INT8 operands: S = Q K^T (forward, and again
// in the backward), O = P V, dV = P^T dO, dQ = dS K, dK = dS^T Q.  dP = dO V^T,
// the product that forms the attention-map gradient, takes FP16 operands.
// Quantization: Q, K, V, dO per head in blocks of 128 tokens, P and dS per
// block of 64 queries x 128 keys, scale amax / 127, codes
// rint(x * (127 / amax)).  The forward is FlashAttention's online softmax
// (P~ = exp(S - running max) quantized per block, the normaliser summed from
// the unquantized P~); the backward recomputes P = exp(S - L) from the saved
// log-sum-exp.
//
// The INT8 products on sm_103a.  Its INT8 tensor rates are far below its
// FP16 ones (the warp-level INT8 MMA runs at a quarter of the FP16 one).  An
// INT8 code is an integer in [-127, 127], exact in FP16; the product of two is
// exact in FP32, and so is every sum of such products below 2^24 (127^2 * 128
// < 2^21 here).  So the six INT8 products run as tcgen05.mma kind::f16 with
// the codes stored as FP16 values, and give the integer results an INT8 MMA
// would (the probes check this on the hardware for every operand form used).
// Each block's integer sum is then scaled by its two block scales in FP32.
//
// Layout.  Every operand lives in the workspace as FP16 rows [token][D] whose
// 16-byte chunks are XOR-permuted by (row & 7) within each 128-byte half: an
// 8-row-aligned run of 128-byte rows is the tensor core's 128-byte-swizzled
// tile, read K-major (D the contraction) or MN-major (tokens the
// contraction).  The codes of Q, dO and V are also stored transposed per
// 64-token tile (V's are the forward's PV operand).
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sagebwd.h"
#include "ptx.cuh"

namespace sagebwd {

using sagefp4::bulk_load;
using sagefp4::globaltimer_ns;
using sagefp4::mbar_arrive_expect_tx;
using sagefp4::mbar_fence_init;
using sagefp4::mbar_init;
using sagefp4::mbar_try_wait;
using sagefp4::smem_addr;
using sagefp4::smem_desc;
using sagefp4::add2;
using sagefp4::fma2;
using sagefp4::hi2;
using sagefp4::lo2;
using sagefp4::max3f;
using sagefp4::mul2;
using sagefp4::pack2;
using sagefp4::tc_commit;
using sagefp4::tc_fence_after;
using sagefp4::tc_fence_before;
using sagefp4::tmem_alloc;
using sagefp4::tmem_dealloc;
using sagefp4::tmem_ld32;
using sagefp4::tmem_relinquish;
using sagefp4::tmem_wait_ld;
using sagefp4::kSwizzle128B;

constexpr int kTok = 128;  // token block of Q, K, V, dO; key tile; key edge of a P / dS block
constexpr int kQ = 64;     // query tile of the backward; query edge of a P / dS block
constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;
constexpr uint64_t kWaitNs = 1500ull * 1000ull * 1000ull;  // bounded copy waits: 1.5 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- layout
// Byte offset of logical (row, byte) in rows W bytes wide (W = 2D: 128 or
// 256): the 16-byte chunk index is XORed with row & 7 (within each 128-byte
// half), the tensor core's 128-byte swizzle; the eight rows of a chunk column
// also fall in eight bank groups.
__host__ __device__ __forceinline__ int swz(int row, int byte, int W) {
  return row * W + ((((byte >> 4) ^ (row & 7))) << 4) + (byte & 15);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_s8(int (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> FP16x2 (lo in the low half), rounded to nearest; exact for
// the integer codes.
__device__ __forceinline__ uint32_t h2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// INT8 code of x in a block with 127 / amax = inv: rint(x * inv) as a float
// (|x| <= amax keeps it within [-127, 127]).
__device__ __forceinline__ float code(float x, float inv) { return rintf(__fmul_rn(x, inv)); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// rint by FP32 arithmetic: (z + 1.5 * 2^23) - 1.5 * 2^23 is z rounded to the
// nearest integer, ties to even, exactly, for |z| < 2^22.
constexpr float kRintMagic = 12582912.0f;

// Warp-wide maximum of unsigned words (every lane gets it).
__device__ __forceinline__ uint32_t redux_max_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Tensor reduction by the copy engine: the box of `map` at (x, y) += the
// shared-memory tile at ssrc (laid out with the map's swizzle), element-wise
// in the map's type, in this thread's bulk group.  wait_read: this thread's
// bulk operations have read their shared-memory sources; wait_all: they have
// completed.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t ssrc, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(ssrc), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

struct Ctl {
  int32_t* status;
  uint64_t limit;
};

// Bounded wait by a whole warp for an mbarrier phase.  False: the copy never
// completed; the status word holds SAGE_FP4_ETIMEOUT.
__device__ __forceinline__ bool waitw(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
    int stop = 0;
    if ((threadIdx.x & 31) == 0 && globaltimer_ns() - t0 > c.limit) {
      atomicCAS(c.status, 0, SAGE_FP4_ETIMEOUT);
      stop = 1;
    }
    if (__shfl_sync(kFull, stop, 0)) return false;
  }
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// -> FP16 bits, rounded to nearest even, saturated to +-65504.
__device__ __forceinline__ uint16_t f2h_sat(float x) {
  x = fminf(fmaxf(x, -65504.0f), 65504.0f);
  return __half_as_ushort(__float2half_rn(x));
}

// ---------------------------------------------------------------- workspace
struct Ws {
  uint16_t *qc, *kc, *vc, *doc;  // INT8 codes as FP16 values, swizzled rows
  uint16_t *vh, *doh;            // V and dO as FP16 values, swizzled rows
  uint16_t *qct, *doct;          // Q^ and dO^ codes transposed: [64-token tile][D][64], swizzled rows
  uint16_t* vct;                 // V^ codes transposed: [128-token tile][2 key halves][D][64], swizzled rows
  float *sq, *sk, *sv, *sdo, *l2, *dd, *dqacc;
  int32_t* status;
};

// ---------------------------------------------------------------- quantizer
// One CTA per (128-token block, head).  kind 0: Q, 1: K, 2: V (codes and the
// FP16 values), 3: dO (codes and FP16 values), with D_i = sum_d dO_id O_id,
// the negated log-sum-exp in log2 units, and dQ's accumulator rows zeroed.
template <int D>
__global__ void __launch_bounds__(kThreads) quant_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v, const uint16_t* __restrict__ o,
                                                         const float* __restrict__ lse, int N, int kind0, Ws ws) {
  __shared__ __align__(16) uint16_t xs[kTok * D];
  __shared__ float red[kThreads / 32];
  const int kind = kind0 + blockIdx.z;
  const int blk = blockIdx.x, bh = blockIdx.y;
  const int nb = (N + kTok - 1) / kTok;
  const int Np = nb * kTok;
  const int n0 = blk * kTok;
  const int rows = min(kTok, N - n0);
  const uint16_t* x = (kind == 1 ? k : kind == 2 ? v : q) + (static_cast<size_t>(bh) * N + n0) * D;
  const int tid = threadIdx.x;

  // load the block (zeros past N) and find its largest magnitude
  float amax = 0.0f;
  constexpr int kVec = kTok * D / 8;  // 16-byte vectors
  for (int i = tid; i < kVec; i += kThreads) {
    const int r = i / (D / 8);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < rows) val = __ldg(reinterpret_cast<const uint4*>(x) + i);
    reinterpret_cast<uint4*>(xs)[i] = val;
    const uint32_t w[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
    }
  }
  amax = warp_max(amax);
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; w++) amax = fmaxf(amax, red[w]);
  const float inv = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
  const size_t hb = static_cast<size_t>(bh) * Np * D;  // this head's first element
  if (tid == 0) {
    float* s = kind == 0 ? ws.sq : kind == 1 ? ws.sk : kind == 2 ? ws.sv : ws.sdo;
    s[static_cast<size_t>(bh) * nb + blk] = __fdiv_rn(amax, 127.0f);
  }
  uint16_t* codes = kind == 0 ? ws.qc : kind == 1 ? ws.kc : kind == 2 ? ws.vc : ws.doc;
  uint16_t* vals = kind == 2 ? ws.vh : ws.doh;
  char* cbase = reinterpret_cast<char*>(codes + hb + static_cast<size_t>(n0) * D);
  char* vbase = reinterpret_cast<char*>(vals + hb + static_cast<size_t>(n0) * D);
  // one 16-byte chunk (8 channels of one row) per step
  for (int i = tid; i < kTok * D / 8; i += kThreads) {
    const int r = i / (D / 8), c = i % (D / 8);
    uint32_t hc[4], hv[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float a = bf2f(xs[r * D + 8 * c + 2 * j]), b = bf2f(xs[r * D + 8 * c + 2 * j + 1]);
      hc[j] = h2(code(a, inv), code(b, inv));
      hv[j] = static_cast<uint32_t>(f2h_sat(a)) | (static_cast<uint32_t>(f2h_sat(b)) << 16);
    }
    const int off = swz(r, 16 * c, 2 * D);
    *reinterpret_cast<uint4*>(cbase + off) = make_uint4(hc[0], hc[1], hc[2], hc[3]);
    if (kind >= 2) *reinterpret_cast<uint4*>(vbase + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
  }
  if (kind == 0 || kind == 2 || kind == 3) {
    // the same codes transposed, per 64-token tile: [D rows][64 tokens], the
    // K-major B operand of dK = dS^T Q and dV = P^T dO, and for V of PV (the
    // two 64-token halves of a 128-token tile are consecutive: [2][D][64])
    uint16_t* tdst = kind == 0 ? ws.qct : kind == 2 ? ws.vct : ws.doct;
    for (int i = tid; i < D * (kTok / 8); i += kThreads) {
      const int d = i % D, c = i / D;  // c: 8-token chunk of the block
      uint32_t h[4];
#pragma unroll
      for (int j = 0; j < 4; j++)
        h[j] = h2(code(bf2f(xs[(8 * c + 2 * j) * D + d]), inv), code(bf2f(xs[(8 * c + 2 * j + 1) * D + d]), inv));
      const int tile = (n0 + 8 * c) / kQ, within = (8 * c) % kQ;
      char* tb = reinterpret_cast<char*>(tdst + hb + static_cast<size_t>(tile) * kQ * D);
      *reinterpret_cast<uint4*>(tb + swz(d, 2 * within, 2 * kQ)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
  }
  if (kind == 3) {
    // D_i = sum_d dO_id O_id and -L in log2 units: one warp per row
    const int warp = tid >> 5, lane = tid & 31;
    for (int r = warp; r < kTok; r += kThreads / 32) {
      float acc = 0.0f;
      if (r < rows) {
        const uint16_t* orow = o + (static_cast<size_t>(bh) * N + n0 + r) * D;
        for (int d = lane; d < D; d += 32) acc = fmaf(bf2f(xs[r * D + d]), bf2f(orow[d]), acc);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
      if (lane == 0) {
        const size_t ix = static_cast<size_t>(bh) * Np + n0 + r;
        ws.dd[ix] = acc;
        ws.l2[ix] = r < rows ? -lse[static_cast<size_t>(bh) * N + n0 + r] * kLog2e : 0.0f;
      }
    }
    float4* acc = reinterpret_cast<float4*>(ws.dqacc + (static_cast<size_t>(bh) * Np + n0) * D);
    for (int i = tid; i < kTok * D / 4; i += kThreads) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ---------------------------------------------------------------- tcgen05
// Instruction descriptor of tcgen05.mma kind::f16: FP16 A and B (formats 0),
// FP32 accumulator (bits 4-5 = 1), both operands K-major, N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A x B^T, FP16 operands in shared memory (descriptors), K = 16.
__device__ __forceinline__ void mma_f16_tc(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Descriptor of a K-major FP16 operand whose rows are 128 bytes (64 values)
// with the 128-byte swizzle (16-byte chunk ^ row & 7), rows of 8 at 1024-byte
// strides, starting k0 values into the row (k0 a multiple of 16); the tile
// must start on a 1024-byte boundary.
// The same with A in tensor memory (M = 128 rows in lanes 0..127; a row's
// K = 16 FP16 values of one step in 8 consecutive 32-bit columns, the lower
// K index in the low half of each column).
__device__ __forceinline__ void mma_f16_tc_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Each thread of the warp writes 32 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ uint64_t desc_k64(uint32_t tile, int k0) {
  return smem_desc(tile + 2 * k0, 16, 1024, kSwizzle128B);
}

// The same products with MN-major operands (idesc bits 15 and 16: A and B
// transposed), as dQ = dS^ K^ reads them: each operand is stored with its K
// index as the 128-byte row (64 FP16 values of M or N per row, 16-byte chunks
// XOR-permuted by row & 7).  The descriptor's leading offset is the distance
// between 64-wide blocks of M (or N), its stride offset the distance between
// groups of 8 K rows (1024 bytes here); a K step of 16 starts 16 rows later.
__host__ __device__ constexpr uint32_t idesc_f16_mn(uint32_t M, uint32_t N) {
  return idesc_f16(M, N) | (1u << 15) | (1u << 16);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int k0, uint32_t block_stride) {
  return smem_desc(tile + 128 * k0, block_stride, 1024, kSwizzle128B);
}

// ---------------------------------------------------------------- backward, tcgen05
// The same backward with all five products on the 5th-generation tensor
// cores, issued asynchronously into tensor memory by one thread while other
// warps work: per 64-query tile the four with 128 keys as rows -- S^T = K^ Q^^T,
// dP^T = V dO^T, dV = P^^T dO^ and dK = dS^^T Q^ (M = 128 keys, N = 64, K = 16
// per instruction) -- and per pair of query tiles dQ = dS^ K^ (M = 128
// queries, N = 64, K = 128 keys) with both operands read MN-major from the
// codes buffers and the resident K^ tile.  The warpgroups of the CTA:
//   0  warp 0: bulk copies; warp 1: tensor-memory allocation and MMA issue
//   1, 2  softmax: each thread owns one key row and half of the tile's 64
//      query columns; P^T and dS^T from the S^T and dP^T rows in tensor
//      memory, their block maxima (one vote of the eight warps each), their
//      INT8 codes written back over S^T and dP^T in tensor memory as the A
//      operands of dV and dK, and dS^T's also to shared memory for dQ
//   3  folds each tile's dV and dK partials (tensor memory) into registers
//      with the tile's block scales, and adds each tile pair's dQ, times its
//      tiles' scales, to the FP32 accumulator in global memory by tensor
//      reductions of the copy engine (staged 32 rows x 32 columns a warp)
// Tensor memory: S^T and dP^T double-buffered (then P^^T and dS^^T in their
// first 32 columns), the dV and dK partials and dQ single, and the resident K^
// and V as the A operands of S^T and dP^T (512 columns); dV and dK read dO^
// and Q^ MN-major from their row tiles.  S^T and dP^T of tile t + 2 are issued
// once dV and dK of tile t have completed.  Every wait is bounded; a wait that runs out
// sets the status word and an abort flag that ends every role's loop.
constexpr int kTcThreads = 512;
constexpr int kTcStages = 3;  // the most stages a tcgen05 kernel uses (mbarrier slots)
struct TcRegs {
  static constexpr uint32_t kCtl = 64, kSoft = 128, kFold = 192;
};
static_assert(TcRegs::kCtl * 128 + TcRegs::kSoft * 256 + TcRegs::kFold * 128 <= 65536, "register split");

template <int D>
struct TcSmem {
  static constexpr int kNH = D / 64;       // 64-wide halves of D
  static constexpr int kTile = 128 * 128;  // 128 rows of 128 bytes
  static constexpr int kK = 0;             // K^ codes [kNH][128 keys][64]
  static constexpr int kV = kNH * kTile;   // FP16 V [kNH][128 keys][64]
  static constexpr int kStageOff = 2 * kNH * kTile;
  // At D = 64 one ring of query tiles, a stage holding Q^ [64 q][64], FP16
  // dO [64 q][64], dO^ [64 q][64], -L and D.  At D = 128 two rings: ring X
  // (S^T and dP^T's operands: Q^ [2][64 q][64], FP16 dO [2][64 q][64]),
  // refilled once those two products are computed, and ring Y (dV and dK's
  // operands: this CTA's halves of Q^ and dO^, [64 q][64] each; -L and D
  // apart, at kLdOff), refilled once dV and dK are.  So the next tiles'
  // copies are not on the path from one tile's dV and dK to the next S^T.
  static constexpr bool kSplit = D == 128;
  static constexpr int kSQ = 0, kSDoh = kNH * 8192, kSDoc = 2 * kNH * 8192, kSL = kSDoc + 8192, kSD = kSL + 256;
  static constexpr int kStage = kSplit ? 2 * kNH * 8192 : (kSD + 256 + 1023) / 1024 * 1024;
  static constexpr int kStages = kSplit ? 2 : 3;
  static constexpr int kYOff = kStageOff + kStages * kStage;
  static constexpr int kYQ = 0, kYDoc = 8192, kYStage = 16384, kYStages = 3;
  static constexpr int kCodesOff = kYOff + (kSplit ? kYStages * kYStage : 0);
  // codes buffers: dS^T [128 keys][64 q] (dQ's A operand, read MN-major),
  // one per tile: two at D = 128, four at D = 64, where the buffer a tile
  // writes was last read by the dQ of tile t - 4's pair, which completed
  // before dV and dK of tile t - 2 and so before this tile's S^T
  static constexpr int kCS = 0, kCodes = kTile, kCodeBufs = kSplit ? 2 : 4;
  // dQ staging: per fold warp a [32 rows][32 FP32] tile, 128-byte swizzled
  static constexpr int kDqOff = kCodesOff + kCodeBufs * kCodes;
  static constexpr int kBarOff = kDqOff + 128 * 128;
  static constexpr int kNumBars = 32;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;  // tmem slot, abort flag, red[2][2][8], scal[4][4]
  static constexpr int kLdOff = kMiscOff + 256;  // ring Y's -L and D: [kYStages][2][64] floats
  static constexpr int kBytes = kLdOff + (kSplit ? kYStages * 512 : 0);
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};
// mbarrier indices
enum {
  TB_FIXED = 0,
  TB_FULL = 1,             // + stage
  TB_EMPTY = 1 + kTcStages,  // + stage
  TB_SDONE = 1 + 2 * kTcStages,  // + buffer (2)
  // + tile mod 4: the tile's codes and scales.  Four slots: the softmax can
  // run up to four tiles ahead of the fold's test (tile t needs only the
  // fold's release of tile t - 3's partials), which with two slots could
  // complete a slot's phase twice before the fold tests it
  TB_CFULL = TB_SDONE + 2,
  TB_CEMPTY = TB_CFULL + 4,
  TB_PDONE = TB_CEMPTY + 2,  // dV and dK partials (single buffer)
  TB_PFREE = TB_PDONE + 1,
  TB_QDONE = TB_PFREE + 1,   // dQ of a tile pair (single buffer)
  TB_QFREE = TB_QDONE + 1,
  TB_KVT = TB_QFREE + 1,     // K^ and V copied into tensor memory
  TB_DRAIN = TB_KVT + 1,
  TB_YFULL = TB_DRAIN + 1,  // + ring Y slot (3, D = 128)
  TB_YEMPTY = TB_YFULL + 3,
  TB_COUNT = TB_YEMPTY + 3
};
static_assert(TB_COUNT <= 32, "barriers");
static_assert(TcSmem<128>::kAlloc <= 227 * 1024, "shared memory");
// tensor-memory columns
constexpr uint32_t kTcS = 0, kTcDp = 128, kTcDv = 256, kTcDk = 320, kTcDq = 384, kTcK = 448, kTcV = 480;

// Bounded warp-wide wait that also gives up when another role has aborted.
__device__ __forceinline__ bool waitw_ab(uint32_t bar, uint32_t parity, const Ctl& c, volatile int* abort) {
  if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
    int stop = 0;
    if ((threadIdx.x & 31) == 0) {
      if (*abort) {
        stop = 1;
      } else if (globaltimer_ns() - t0 > c.limit) {
        *abort = 1;
        atomicCAS(c.status, 0, SAGE_FP4_ETIMEOUT);
        stop = 1;
      }
    }
    if (__shfl_sync(kFull, stop, 0)) return false;
  }
}

// The same for a single thread.
// Two bounded waits by a whole warp with one vote when both phases have
// completed already (the usual case), else one after the other.
__device__ __forceinline__ bool waitw2_ab(uint32_t bar0, uint32_t par0, uint32_t bar1, uint32_t par1, const Ctl& c,
                                          volatile int* abort) {
  if (__all_sync(kFull, mbar_try_wait(bar0, par0) && mbar_try_wait(bar1, par1))) return true;
  return waitw_ab(bar0, par0, c, abort) && waitw_ab(bar1, par1, c, abort);
}
__device__ __forceinline__ bool wait1_ab(uint32_t bar, uint32_t parity, const Ctl& c, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > c.limit) {
      *abort = 1;
      atomicCAS(c.status, 0, SAGE_FP4_ETIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive1(uint32_t bar) { sagefp4::mbar_arrive(bar); }

// One lane of the (converged) warp: true there, false elsewhere.  The MMA
// issuers run as whole warps, so their descriptors and loop state are
// warp-uniform, and the elected lane issues.
__device__ __forceinline__ bool elect1() {
  uint32_t p;
  asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}" : "=r"(p));
  return p != 0;
}

// All 256 threads of the two softmax warpgroups: AND of `ok` over them
// (named barrier 1).
__device__ __forceinline__ bool group_and(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.and.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(ok))
      : "memory");
  return r != 0;
}

// Each thread of the warp reads 16 consecutive FP32 columns of its lane.
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  sagefp4::tmem_ld16(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// Tensor maps of the backward.  dq: the FP32 dQ accumulator [B*H*Np][D]
// (boxes of 32 x 32, 128-byte swizzled).  At D = 128 also k, v: K^ codes and
// FP16 V as bytes [B*H*Np][256], boxes of 128 bytes x 128 rows; q, doh, doc:
// Q^ codes, FP16 dO and dO^ codes, boxes of 128 bytes x 64 rows (the rows'
// 16-byte chunks are XOR-permuted within each 128-byte half, so a copied half
// is in the 128-byte-swizzled layout).
struct BwdMaps {
  CUtensorMap dq, k, v, q, doh, doc;
};

template <int D, bool kCausal>
__global__ void __launch_bounds__(kTcThreads, 1)
    dkdv_tc_kernel(const __grid_constant__ BwdMaps maps, Ws ws, uint16_t* __restrict__ dk,
                   uint16_t* __restrict__ dv, int N, float scale, uint64_t wait_ns, int withhold) {
  using L = TcSmem<D>;
  constexpr int kSt = L::kStages, kYSt = L::kYStages;
  constexpr bool kSplit = L::kSplit;
  // The grid is (key tiles, heads, halves of D), dispatched in that order
  // (x fastest); its linear index is mapped to (key tile, head, half) with
  // the key tile slowest, so that in the causal case the CTAs with the most
  // query tiles (the first key tiles) start first over all heads (simulated
  // makespan 6.5% shorter than dispatching every head's tiles in turn)
  const int lin = static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  const int dh = lin % static_cast<int>(gridDim.z);  // this CTA's 64 columns of dV, dK, dQ
  const int kb = lin / static_cast<int>(gridDim.z * gridDim.y);
  const int bh = lin / static_cast<int>(gridDim.z) % static_cast<int>(gridDim.y);
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, by pointer arithmetic on the shared array (so
  // that the compiler keeps its accesses in the shared state space)
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const int nkt = (N + kTok - 1) / kTok;
  const int Np = nkt * kTok;
  const int nqt = Np / kQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wg = warp >> 2;
  const size_t hb = static_cast<size_t>(bh) * Np * D;
  const size_t hrow = static_cast<size_t>(bh) * Np;
  const int q0 = kCausal ? 2 * kb : 0;
  const int niter = nqt - q0;
  const Ctl ctl{ws.status, wait_ns};
  auto bar = [&](int i) { return sbase + L::kBarOff + 8 * i; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  float* red = reinterpret_cast<float*>(smem + L::kMiscOff + 16);    // [2 parity][2 kinds][8 warps]
  float* scal = reinterpret_cast<float*>(smem + L::kMiscOff + 160);  // [tile mod 4][4]

  if (threadIdx.x == 0) {
    mbar_init(bar(TB_FIXED), 1);
    for (int s = 0; s < kSt; s++) {
      mbar_init(bar(TB_FULL + s), 1);
      mbar_init(bar(TB_EMPTY + s), kSplit ? 1 : 1 + 8);  // the MMA commit (+ the softmax warps: -L, D)
    }
    for (int s = 0; s < (kSplit ? kYSt : 0); s++) {
      mbar_init(bar(TB_YFULL + s), 1);
      mbar_init(bar(TB_YEMPTY + s), 1 + 8);  // the MMA commit + the softmax warps
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(bar(TB_SDONE + b), 1);
      mbar_init(bar(TB_CEMPTY + b), 1);  // the MMA commit after the pair's dQ
    }
    for (int q = 0; q < 4; q++) mbar_init(bar(TB_CFULL + q), 8);
    mbar_init(bar(TB_PDONE), 1);
    mbar_init(bar(TB_PFREE), 4);
    mbar_init(bar(TB_QDONE), 1);
    mbar_init(bar(TB_QFREE), 4);
    mbar_init(bar(TB_KVT), 4);
    mbar_init(bar(TB_DRAIN), 1);
    *abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (wg == 0) {
    sagefp4::regs_dec<TcRegs::kCtl>();
    if (kSplit && warp == 2 && lane == 0) {
      // ---- producer of ring Y (D = 128)
      const int hr = static_cast<int>(hrow);
      int issued = 0;
      for (int it = 0; it < niter; it++) {
        const int y = it % kYSt;
        if (it >= kYSt && !wait1_ab(bar(TB_YEMPTY + y), ((it / kYSt) - 1) & 1, ctl, abort)) break;
        const int qtile = q0 + it;
        const uint32_t yb = sbase + L::kYOff + y * L::kYStage, ld = sbase + L::kLdOff + y * 512;
        mbar_arrive_expect_tx(bar(TB_YFULL + y), 2 * 8192 + 512);
        sagefp4::tma_load_2d(yb + L::kYQ, &maps.q, 128 * dh, hr + qtile * kQ, bar(TB_YFULL + y));
        sagefp4::tma_load_2d(yb + L::kYDoc, &maps.doc, 128 * dh, hr + qtile * kQ, bar(TB_YFULL + y));
        bulk_load(ld, ws.l2 + hrow + static_cast<size_t>(qtile) * kQ, 256, bar(TB_YFULL + y));
        bulk_load(ld + 256, ws.dd + hrow + static_cast<size_t>(qtile) * kQ, 256, bar(TB_YFULL + y));
        issued = it + 1;
      }
      if (*abort) {
        for (int last = issued - 1; last >= 0 && last >= issued - kYSt; last--) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar(TB_YFULL + last % kYSt), (last / kYSt) & 1) && globaltimer_ns() - t0 < ctl.limit) {
          }
        }
      }
    } else if (warp == 0 && lane == 0) {
      // ---- producer (of ring X at D = 128)
      const int hr = static_cast<int>(hrow);  // the head's first row in [B*H*Np]
      mbar_arrive_expect_tx(bar(TB_FIXED), 2 * L::kNH * L::kTile);
      if constexpr (D == 64) {
        const size_t off = hb + static_cast<size_t>(kb) * kTok * D;
        bulk_load(sbase + L::kK, ws.kc + off, L::kTile, bar(TB_FIXED));
        bulk_load(sbase + L::kV, ws.vh + off, L::kTile, bar(TB_FIXED));
      } else {
        for (int x = 0; x < 2; x++) {
          sagefp4::tma_load_2d(sbase + L::kK + x * L::kTile, &maps.k, 128 * x, hr + kb * kTok, bar(TB_FIXED));
          sagefp4::tma_load_2d(sbase + L::kV + x * L::kTile, &maps.v, 128 * x, hr + kb * kTok, bar(TB_FIXED));
        }
      }
      const bool held = withhold && lin == 0;
      int issued = 0;
      for (int it = 0; it < niter; it++) {
        const int s = it % kSt;
        if (it >= kSt && !wait1_ab(bar(TB_EMPTY + s), ((it / kSt) - 1) & 1, ctl, abort)) break;
        if (held && it == 0) continue;  // failure-detection test: this tile never arrives
        const int qtile = q0 + it;
        const uint32_t st = sbase + L::kStageOff + s * L::kStage;
        mbar_arrive_expect_tx(bar(TB_FULL + s), kSplit ? L::kStage : (2 * L::kNH + 1) * 8192 + 512);
        if constexpr (D == 64) {
          const size_t qo = hb + static_cast<size_t>(qtile) * kQ * D;
          bulk_load(st + L::kSQ, ws.qc + qo, 8192, bar(TB_FULL + s));
          bulk_load(st + L::kSDoh, ws.doh + qo, 8192, bar(TB_FULL + s));
          bulk_load(st + L::kSDoc, ws.doc + qo, 8192, bar(TB_FULL + s));
        } else {
          const int r = hr + qtile * kQ;
          for (int x = 0; x < 2; x++) {
            sagefp4::tma_load_2d(st + L::kSQ + 8192 * x, &maps.q, 128 * x, r, bar(TB_FULL + s));
            sagefp4::tma_load_2d(st + L::kSDoh + 8192 * x, &maps.doh, 128 * x, r, bar(TB_FULL + s));
          }
        }
        if constexpr (!kSplit) {
          bulk_load(st + L::kSL, ws.l2 + hrow + static_cast<size_t>(qtile) * kQ, 256, bar(TB_FULL + s));
          bulk_load(st + L::kSD, ws.dd + hrow + static_cast<size_t>(qtile) * kQ, 256, bar(TB_FULL + s));
        }
        issued = it + 1;
      }
      if (*abort) {
        // let every copy this thread issued land before the CTA exits
        for (int last = issued - 1; last >= 0 && last >= issued - kSt; last--)
          if (!(held && last == 0)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar(TB_FULL + last % kSt), (last / kSt) & 1) && globaltimer_ns() - t0 < ctl.limit) {
            }
          }
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar(TB_FIXED), 0) && globaltimer_ns() - t0 < ctl.limit) {
        }
      }
    } else if (warp == 1) {
      // ---- MMA issue: the whole warp, one elected lane issues
      // B MN-major for dV and dK (dO^ and Q^ as [64 q][64 d] rows)
      const uint32_t id = idesc_f16(128, 64), idb = idesc_f16(128, 64) | (1u << 16), idq = idesc_f16_mn(128, 64);
      // dQ = dS^ K^, MN-major: a K step of 16 rows moves 2048 bytes (+128);
      // K^'s 64 columns of this CTA's half
      const uint64_t dqa = desc_mn(sbase + L::kCodesOff + L::kCS, 0, L::kCodes);
      const uint64_t dqb = desc_mn(sbase + L::kK + dh * L::kTile, 0, L::kCodes);
      // S^T and dP^T at D = 128: K^ and V from shared memory (a 64-wide half
      // is 16 KB, +1024)
      const uint64_t dk0 = desc_k64(sbase + L::kK, 0), dv0 = desc_k64(sbase + L::kV, 0);
      bool ok = waitw_ab(bar(TB_FIXED), 0, ctl, abort) && (D != 64 || waitw_ab(bar(TB_KVT), 0, ctl, abort));
      auto issue_sdp = [&](int it) {
        const int s = it % kSt, b = it & 1;
        if (!waitw_ab(bar(TB_FULL + s), (it / kSt) & 1, ctl, abort)) return false;
        // buffer b: dV and dK of tile it - 2 have read its P^^T and dS^^T (the
        // latest completion of PDONE can be tile it - 2's: tile it - 1's dV and
        // dK are issued after this)
        if (it >= 2 && !waitw_ab(bar(TB_PDONE), (it - 2) & 1, ctl, abort)) return false;
        tc_fence_after();
        const uint32_t st = sbase + L::kStageOff + s * L::kStage;
        // descriptors built once per operand; a K step of 16 moves 32 bytes
        // (+2), a 64-wide half of Q^ or dO (64 rows) 8 KB (+512)
        const uint64_t dq = desc_k64(st + L::kSQ, 0), ddo = desc_k64(st + L::kSDoh, 0);
        if (elect1()) {
          if constexpr (D == 64) {
#pragma unroll
            for (int k = 0; k < 4; k++) mma_f16_tc_ta(tmem + kTcS + 64 * b, tmem + kTcK + 8 * k, dq + 2 * k, id, k > 0);
#pragma unroll
            for (int k = 0; k < 4; k++)
              mma_f16_tc_ta(tmem + kTcDp + 64 * b, tmem + kTcV + 8 * k, ddo + 2 * k, id, k > 0);
          } else {
#pragma unroll
            for (int k = 0; k < D / 16; k++)
              mma_f16_tc(tmem + kTcS + 64 * b, dk0 + 1024 * (k >> 2) + 2 * (k & 3), dq + 512 * (k >> 2) + 2 * (k & 3),
                         id, k > 0);
#pragma unroll
            for (int k = 0; k < D / 16; k++)
              mma_f16_tc(tmem + kTcDp + 64 * b, dv0 + 1024 * (k >> 2) + 2 * (k & 3),
                         ddo + 512 * (k >> 2) + 2 * (k & 3), id, k > 0);
          }
          tc_commit(bar(TB_SDONE + b));
          if constexpr (kSplit) tc_commit(bar(TB_EMPTY + s));
        }
        __syncwarp();
        return true;
      };
      if (ok) ok = issue_sdp(0);
      for (int it = 0; ok && it < niter; it++) {
        const int s = it % kSt, b = it & 1;
        if (it + 1 < niter && !(ok = issue_sdp(it + 1))) break;
        if (!(ok = waitw_ab(bar(TB_CFULL + (it & 3)), (it >> 2) & 1, ctl, abort))) break;
        if (b == 1) {
          // dQ of the pair (it - 1, it) first -- rows 0..63 from the codes
          // buffer of tile it - 1, rows 64..127 from tile it's, their only
          // reader -- so that the buffers are released for later tiles'
          // codes early; the fold has read the previous pair's dQ.  With four
          // buffers pair pr reads buffers 2 (pr & 1) and 2 (pr & 1) + 1.
          const int pr = it >> 1;
          if (pr >= 1 && !(ok = waitw_ab(bar(TB_QFREE), (pr - 1) & 1, ctl, abort))) break;
          tc_fence_after();
          const uint64_t dqp = dqa + (L::kCodeBufs == 4 && (pr & 1) ? (2 * L::kCodes) >> 4 : 0);
          if (elect1()) {
#pragma unroll
            for (int k = 0; k < 8; k++) mma_f16_tc(tmem + kTcDq, dqp + 128 * k, dqb + 128 * k, idq, k > 0);
            tc_commit(bar(TB_QDONE));
            if constexpr (L::kCodeBufs == 2) {
              tc_commit(bar(TB_CEMPTY + 0));
              tc_commit(bar(TB_CEMPTY + 1));
            }
          }
          __syncwarp();
        }
        // the partials' buffer: the fold has read the previous tile's
        if (it >= 1 && !(ok = waitw_ab(bar(TB_PFREE), (it - 1) & 1, ctl, abort))) break;
        const int y = kSplit ? it % kYSt : 0;
        if (kSplit && !(ok = waitw_ab(bar(TB_YFULL + y), (it / kYSt) & 1, ctl, abort))) break;
        tc_fence_after();
        // B: this CTA's 64 columns of dO^ and Q^, MN-major
        const uint32_t st = sbase + L::kStageOff + s * L::kStage, yb = sbase + L::kYOff + y * L::kYStage;
        const uint64_t ddoc = kSplit ? desc_mn(yb + L::kYDoc, 0, 8192) : desc_mn(st + L::kSDoc, 0, 8192);
        const uint64_t dqm = kSplit ? desc_mn(yb + L::kYQ, 0, 8192) : desc_mn(st + L::kSQ + 8192 * dh, 0, 8192);
        // A: P^^T and dS^^T in tensor memory (8 columns a K step of 16 queries)
        if (elect1()) {
#pragma unroll
          for (int k = 0; k < 4; k++)
            mma_f16_tc_ta(tmem + kTcDv, tmem + kTcS + 64 * b + 8 * k, ddoc + 128 * k, idb, k > 0);
#pragma unroll
          for (int k = 0; k < 4; k++)
            mma_f16_tc_ta(tmem + kTcDk, tmem + kTcDp + 64 * b + 8 * k, dqm + 128 * k, idb, k > 0);
          tc_commit(bar(TB_PDONE));
          tc_commit(bar(kSplit ? TB_YEMPTY + y : TB_EMPTY + s));
        }
        __syncwarp();
      }
      // every MMA issued has completed before tensor memory is released
      if (elect1()) tc_commit(bar(TB_DRAIN));
      __syncwarp();
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar(TB_DRAIN), 0) && globaltimer_ns() - t0 < ctl.limit) {
      }
    }
  } else if (wg == 1 || wg == 2) {
    // ---- softmax: this thread's key row, query columns 32h..32h+31
    sagefp4::regs_inc<TcRegs::kSoft>();
    const int h = wg - 1;
    const int row = 32 * (warp & 3) + lane;     // 0..127
    const int sw = 4 * h + (warp & 3);          // softmax warp 0..7
    const uint32_t lanebase = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int key = kb * kTok + row;
    const float sk = ws.sk[static_cast<size_t>(bh) * nkt + kb];
    const float c2base = sk * scale * kLog2e;
    // the query tile's block scales, read one tile ahead
    float sq_next = ws.sq[static_cast<size_t>(bh) * nkt + (q0 >> 1)];
    float sdo_next = ws.sdo[static_cast<size_t>(bh) * nkt + (q0 >> 1)];
    for (int it = 0; it < niter; it++) {
      const int s = it % kSt, b = it & 1, qtile = q0 + it;
      const float sq = sq_next, sdo = sdo_next;
      if (it + 1 < niter) {
        sq_next = ws.sq[static_cast<size_t>(bh) * nkt + ((qtile + 1) >> 1)];
        sdo_next = ws.sdo[static_cast<size_t>(bh) * nkt + ((qtile + 1) >> 1)];
      }
      // a failed wait is voted on below, before anything is published
      const int y = kSplit ? it % kYSt : 0;
      bool ok = kSplit ? waitw2_ab(bar(TB_SDONE + b), (it >> 1) & 1, bar(TB_YFULL + y), (it / kYSt) & 1, ctl, abort)
                       : waitw2_ab(bar(TB_SDONE + b), (it >> 1) & 1, bar(TB_FULL + s), (it / kSt) & 1, ctl, abort);
      tc_fence_after();
      // this half of the S^T and dP^T rows: two loads in flight, one wait
      uint32_t ru[2][32];
      tmem_ld32(tmem + lanebase + kTcS + 64 * b + 32 * h, ru[0]);
      tmem_ld32(tmem + lanebase + kTcDp + 64 * b + 32 * h, ru[1]);
      tmem_wait_ld();
      float p[32], dp[32];
#pragma unroll
      for (int i = 0; i < 32; i++) {
        p[i] = __uint_as_float(ru[0][i]);
        dp[i] = __uint_as_float(ru[1][i]);
      }
      // P^T = exp2(S^T c - L); masked and padded entries 0; dS^T = P^T o (dP^T - D)
      const float* Ls = reinterpret_cast<const float*>(kSplit ? smem + L::kLdOff + y * 512
                                                              : smem + L::kStageOff + s * L::kStage + L::kSL) + 32 * h;
      const float* Ds = Ls + 64;
      const float c2 = c2base * sq;
      const bool edge = (kCausal && qtile <= 2 * kb + 1) || (qtile * kQ + kQ > N) || (kb * kTok + kTok > N);
      // (pairs of columns through the packed FP32 forms, each lane rounded
      // like its scalar form; Ls holds -L)
      float pmax = 0.0f, smax = 0.0f;
      const uint64_t cc = pack2(c2, c2);
#pragma unroll
      for (int q4 = 0; q4 < 8; q4++) {
        const float4 l4 = reinterpret_cast<const float4*>(Ls)[q4];
        const float4 d4 = reinterpret_cast<const float4*>(Ds)[q4];
        const uint64_t l01 = pack2(l4.x, l4.y), l23 = pack2(l4.z, l4.w);
        const int q = 4 * q4;
        const uint64_t x01 = fma2(pack2(p[q], p[q + 1]), cc, l01), x23 = fma2(pack2(p[q + 2], p[q + 3]), cc, l23);
        float v[4] = {ex2(lo2(x01)), ex2(hi2(x01)), ex2(lo2(x23)), ex2(hi2(x23))};
        if (edge) {
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const int query = qtile * kQ + 32 * h + q + e;
            if (query >= N || key >= N || (kCausal && key > query)) v[e] = 0.0f;
          }
        }
        const uint64_t s01 = mul2(pack2(v[0], v[1]), add2(pack2(dp[q], dp[q + 1]), pack2(-d4.x, -d4.y)));
        const uint64_t s23 = mul2(pack2(v[2], v[3]), add2(pack2(dp[q + 2], dp[q + 3]), pack2(-d4.z, -d4.w)));
        p[q] = v[0];
        p[q + 1] = v[1];
        p[q + 2] = v[2];
        p[q + 3] = v[3];
        dp[q] = lo2(s01);
        dp[q + 1] = hi2(s01);
        dp[q + 2] = lo2(s23);
        dp[q + 3] = hi2(s23);
        pmax = max3f(pmax, max3f(v[0], v[1], v[2]), v[3]);
        smax = max3f(smax, max3f(fabsf(dp[q]), fabsf(dp[q + 1]), fabsf(dp[q + 2])), fabsf(dp[q + 3]));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive1(bar(kSplit ? TB_YEMPTY + y : TB_EMPTY + s));  // L and D read
      // both maxima are >= 0 (or -0): the warp maximum of their bit patterns
      // with the sign bit cleared
      const uint32_t pm = redux_max_u32(__float_as_uint(pmax) & 0x7fffffffu);
      const uint32_t sm = redux_max_u32(__float_as_uint(smax) & 0x7fffffffu);
      if (lane == 0) {
        red[(b * 2 + 0) * 8 + sw] = __uint_as_float(pm);
        red[(b * 2 + 1) * 8 + sw] = __uint_as_float(sm);
      }
      // with two codes buffers, this tile's is free once the pair's dQ (tiles
      // it - 2, it - 1) has read it; the vote below also orders both halves'
      // tensor-memory loads before the codes overwrite them
      if constexpr (L::kCodeBufs == 2)
        ok = ok && (it < 2 || waitw_ab(bar(TB_CEMPTY + b), ((it >> 1) - 1) & 1, ctl, abort));
      if (!group_and(ok)) break;  // also publishes red[]
      const float4* r4 = reinterpret_cast<const float4*>(red + b * 16);
      const float4 p0 = r4[0], p1 = r4[1], s0 = r4[2], s1 = r4[3];
      const float pa = fmaxf(max3f(max3f(p0.x, p0.y, p0.z), max3f(p0.w, p1.x, p1.y), p1.z), p1.w);
      const float sa = fmaxf(max3f(max3f(s0.x, s0.y, s0.z), max3f(s0.w, s1.x, s1.y), s1.z), s1.w);
      const float pinv = pa > 0.0f ? __fdiv_rn(127.0f, pa) : 0.0f;
      const float sinv = sa > 0.0f ? __fdiv_rn(127.0f, sa) : 0.0f;
      uint8_t* cbuf = smem + L::kCodesOff + (it % L::kCodeBufs) * L::kCodes;
      const uint64_t pp = pack2(pinv, pinv), ss = pack2(sinv, sinv);
      // rint(x * inv) for a pair, as FP16x2: x * inv + 1.5 * 2^23 in one FMA
      // rounds the exact product to an integer (ties to even), and
      // subtracting 1.5 * 2^23 is exact
      const uint64_t magic2 = pack2(kRintMagic, kRintMagic), nmagic2 = pack2(-kRintMagic, -kRintMagic);
      auto code2 = [&](float a, float b, uint64_t inv2) {
        const uint64_t y = add2(fma2(pack2(a, b), inv2, magic2), nmagic2);
        return h2(lo2(y), hi2(y));
      };
      // codes of query columns 2j, 2j + 1 of this half in word j: P^^T and
      // dS^^T over the first 32 columns of S^T and dP^T (tensor memory),
      // dS^^T also to shared memory
      uint32_t wp[16], wsd[16];
#pragma unroll
      for (int j = 0; j < 16; j++) {
        wp[j] = code2(p[2 * j], p[2 * j + 1], pp);
        wsd[j] = code2(dp[2 * j], dp[2 * j + 1], ss);
      }
      tmem_st16(tmem + lanebase + kTcS + 64 * b + 16 * h, wp);
      tmem_st16(tmem + lanebase + kTcDp + 64 * b + 16 * h, wsd);
#pragma unroll
      for (int ch = 0; ch < 4; ch++)
        *reinterpret_cast<uint4*>(cbuf + L::kCS + swz(row, 64 * h + 16 * ch, 128)) =
            make_uint4(wsd[4 * ch], wsd[4 * ch + 1], wsd[4 * ch + 2], wsd[4 * ch + 3]);
      tmem_wait_st();
      if (threadIdx.x == 128) {
        float* sc = scal + 4 * (it & 3);
        if constexpr (kSplit) {
          // the block maxima; the fold forms the scales (measured 4% faster
          // at D = 128, 4% slower at D = 64)
          sc[0] = pa;
          sc[1] = sa;
        } else {
          const float sp = __fdiv_rn(pa, 127.0f), sds = __fdiv_rn(sa, 127.0f);
          sc[0] = sp * sdo;          // dV
          sc[1] = sds * sq;          // dK (the softmax scale comes at the end)
          sc[2] = sds * sk * scale;  // dQ
        }
      }
      // the codes (tensor-memory stores; generic-proxy shared-memory writes) ->
      // visible to the tensor core
      tc_fence_before();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive1(bar(TB_CFULL + (it & 3)));
    }
  } else {
    // ---- dV and dK folds, and dQ read out (warpgroup 3)
    sagefp4::regs_inc<TcRegs::kFold>();
    const int row = 32 * (warp & 3) + lane;  // key row of the folds; query row of a tile pair's dQ
    const uint32_t lanebase = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    uint64_t accv[32], acck[32];  // FP32 pairs
#pragma unroll
    for (int i = 0; i < 32; i++) accv[i] = acck[i] = 0;
    float fq[2] = {0.0f, 0.0f};  // dQ scales of the pair's two tiles
    // D = 64: K^ and V rows (this thread's key) into tensor memory, the A
    // operands of S^T and dP^T for the CTA's whole life
    bool kv_ok = D != 64 || waitw_ab(bar(TB_FIXED), 0, ctl, abort);
    if (D == 64 && kv_ok) {
#pragma unroll
      for (int which = 0; which < 2; which++) {
        uint32_t w[32];
        const uint8_t* src = smem + (which == 0 ? L::kK : L::kV);
#pragma unroll
        for (int c = 0; c < 8; c++) {
          const uint4 v4 = *reinterpret_cast<const uint4*>(src + swz(row, 16 * c, 128));
          w[4 * c] = v4.x;
          w[4 * c + 1] = v4.y;
          w[4 * c + 2] = v4.z;
          w[4 * c + 3] = v4.w;
        }
        tmem_st32(tmem + lanebase + (which == 0 ? kTcK : kTcV), w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(bar(TB_KVT));
    }
    // D = 128: the block scales of K (this CTA's keys) and, one tile ahead,
    // of Q and dO
    const float skf = kSplit ? ws.sk[static_cast<size_t>(bh) * nkt + kb] : 0.0f;
    float sq_next = kSplit ? ws.sq[static_cast<size_t>(bh) * nkt + (q0 >> 1)] : 0.0f;
    float sdo_next = kSplit ? ws.sdo[static_cast<size_t>(bh) * nkt + (q0 >> 1)] : 0.0f;
    for (int it = 0; kv_ok && it < niter; it++) {
      const int b = it & 1;
      // CFULL: this tile's block scales (D = 128: block maxima) are written
      if (!waitw_ab(bar(TB_CFULL + (it & 3)), (it >> 2) & 1, ctl, abort)) break;
      const float* sc = scal + 4 * (it & 3);
      uint64_t fv, fk;
      if constexpr (kSplit) {
        const float sqf = sq_next, sdof = sdo_next;
        if (it + 1 < niter) {
          sq_next = ws.sq[static_cast<size_t>(bh) * nkt + ((q0 + it + 1) >> 1)];
          sdo_next = ws.sdo[static_cast<size_t>(bh) * nkt + ((q0 + it + 1) >> 1)];
        }
        const float sp = __fdiv_rn(sc[0], 127.0f), sds = __fdiv_rn(sc[1], 127.0f);
        const float cv = sp * sdof;  // dV
        const float ck = sds * sqf;  // dK (the softmax scale comes at the end)
        fv = pack2(cv, cv);
        fk = pack2(ck, ck);
        fq[b] = sds * skf * scale;  // dQ
      } else {
        fv = pack2(sc[0], sc[0]);
        fk = pack2(sc[1], sc[1]);
        fq[b] = sc[2];
      }
      if (!waitw_ab(bar(TB_PDONE), it & 1, ctl, abort)) break;
      tc_fence_after();
#pragma unroll
      for (int qc = 0; qc < 4; qc++) {
        uint32_t rv[16], rk[16];
        sagefp4::tmem_ld16(tmem + lanebase + kTcDv + 16 * qc, rv);
        sagefp4::tmem_ld16(tmem + lanebase + kTcDk + 16 * qc, rk);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; i++) {
          accv[8 * qc + i] = fma2(pack2(__uint_as_float(rv[2 * i]), __uint_as_float(rv[2 * i + 1])), fv, accv[8 * qc + i]);
          acck[8 * qc + i] = fma2(pack2(__uint_as_float(rk[2 * i]), __uint_as_float(rk[2 * i + 1])), fk, acck[8 * qc + i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(bar(TB_PFREE));
      if (b == 1) {
        // dQ rows of query tiles it - 1 (rows 0..63) and it (64..127)
        if (!waitw_ab(bar(TB_QDONE), (it >> 1) & 1, ctl, abort)) break;
        tc_fence_after();
        const float f = row < kQ ? fq[0] : fq[1];
        const uint64_t f2 = pack2(f, f);
        // this warp's rows of the pair in the accumulator viewed as [B*H*Np][64]
        const int y0 = static_cast<int>(hrow) + (q0 + it - 1) * kQ + 32 * (warp & 3);
        uint8_t* wt = smem + L::kDqOff + 4096 * (warp & 3);
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          uint32_t r[32];
          tmem_ld32(tmem + lanebase + kTcDq + 32 * hh, r);
          if (lane == 0) bulk_wait_read();  // the staging tile's previous reduction has read it
          __syncwarp();
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 8; c++) {
            const uint64_t x01 = mul2(pack2(__uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1])), f2);
            const uint64_t x23 = mul2(pack2(__uint_as_float(r[4 * c + 2]), __uint_as_float(r[4 * c + 3])), f2);
            *reinterpret_cast<uint4*>(wt + swz(lane, 16 * c, 128)) =
                make_uint4(static_cast<uint32_t>(x01), static_cast<uint32_t>(x01 >> 32), static_cast<uint32_t>(x23),
                           static_cast<uint32_t>(x23 >> 32));
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_2d(&maps.dq, smem_addr(wt), 64 * dh + 32 * hh, y0);
            bulk_commit();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive1(bar(TB_QFREE));
      }
    }
    if (lane == 0) bulk_wait_all();  // the dQ reductions have read shared memory and completed
    __syncwarp();
    if (!*abort) {
      const int key = kb * kTok + row;
      if (key < N) {
#pragma unroll
        for (int which = 0; which < 2; which++) {
          uint16_t* dst = (which == 0 ? dv : dk) + (static_cast<size_t>(bh) * N + key) * D + 64 * dh;
          const float f = which == 0 ? 1.0f : scale;
          const uint64_t* acc = which == 0 ? accv : acck;
#pragma unroll
          for (int c = 0; c < 8; c++) {
            uint4 w;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(lo2(acc[4 * c + 0]) * f, hi2(acc[4 * c + 0]) * f);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(lo2(acc[4 * c + 1]) * f, hi2(acc[4 * c + 1]) * f);
            __nv_bfloat162 h2v = __floats2bfloat162_rn(lo2(acc[4 * c + 2]) * f, hi2(acc[4 * c + 2]) * f);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(lo2(acc[4 * c + 3]) * f, hi2(acc[4 * c + 3]) * f);
            w.x = *reinterpret_cast<uint32_t*>(&h0);
            w.y = *reinterpret_cast<uint32_t*>(&h1);
            w.z = *reinterpret_cast<uint32_t*>(&h2v);
            w.w = *reinterpret_cast<uint32_t*>(&h3);
            *reinterpret_cast<uint4*>(dst + 8 * c) = w;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- forward, tcgen05
// The forward with S = Q^ K^^T and O_t = P~^ V^ on the 5th-generation tensor
// cores (M = 128 query rows; S: N = 128 keys; PV: N = 64), issued by one
// thread into double-buffered tensor memory.  A persistent CTA walks a fixed
// list of work items, one 128-query tile of one head each (causal: the
// longest first); the KV tiles of its items form one stream g = 0, 1, ...
// that every role walks in the same order, so the next item's first tiles
// overlap the current item's last ones and its epilogue.  The warpgroups:
//   0  warp 0: bulk copies of Q^ (two slots, by item) and K^; warp 1:
//      tensor-memory allocation and MMA issue; warp 2: bulk copies of V^T
//      (at D = 128)
//   1, 2  softmax: each thread owns one query row and 64 of the tile's 128
//      keys; the row maximum and the 64-row block maxima are exchanged
//      through shared memory; P~'s INT8 codes go to tensor memory (tcgen05.st)
//      as the A operand of PV, each warpgroup writing its 64 keys
//   3  correction: O in registers, rescaled by each row's factor and
//      accumulated with each tile's PV times its block scales; each item's
//      epilogue once the softmax has published the item's l and m
// P~ blocks are 64 query rows x 128 keys, as in the warp-level forward.
template <int D>
struct TfSmem {
  static constexpr int kHalf = 128 * 128;          // 128 rows of 128 bytes
  static constexpr int kQBytes = D / 64 * kHalf;   // Q^ [D / 64 halves][128][64]
  static constexpr int kQ = 0;                     // two Q^ slots, by item
  static constexpr int kStageOff = 2 * kQBytes;
  static constexpr int kSK = 0;                    // K^ [D / 64 halves][128 keys][64]
  static constexpr int kSV = D / 64 * kHalf;       // V^T [2 key halves][D][64 keys]
  static constexpr int kStage = 2 * D / 64 * kHalf;
  static constexpr int kStages = D == 64 ? 3 : 2;
  static constexpr int kBarOff = kStageOff + kStages * kStage;
  static constexpr int kMiscOff = kBarOff + 8 * 32;
  // misc: tmem slot, abort, row max halves [2 parity][2][128], alpha [tile
  // mod 4][128], block max [2 parity][8 warps], beta [tile mod 4][2], final l
  // halves [2 item slots][2][128], m [2 item slots][128]
  static constexpr int kXm = kMiscOff + 16, kAl = kXm + 2048, kBm = kAl + 2048, kBeta = kBm + 64,
                       kLf = kBeta + 32, kMf = kLf + 2048;
  static constexpr int kBytes = kMf + 1024;
  static constexpr int kAlloc = kBytes + 1024;
};
static_assert(TfSmem<128>::kAlloc <= 227 * 1024, "shared memory");
// mbarriers (3 stages at most); K^ and V^T of a stage fill and empty
// separately: K^ is free once S has been computed, V^T once PV has
enum {
  FB_Q = 0,        // + item slot (2): Q^ landed
  FB_QEMPTY = 2,   // + item slot: every S of the slot's item completed
  FB_KFULL = 4,
  FB_VFULL = 7,
  FB_KEMPTY = 10,
  FB_VEMPTY = 13,
  FB_SDONE = 16,  // + buffer
  // + tile mod 4: P^, alpha and beta of the tile.  Four slots: the softmax
  // can run up to four tiles ahead of the correction (tile t needs only the
  // correction's release of PV of tile t - 4), which with two slots could
  // complete a slot's phase twice before the correction tests it
  FB_PFULL = FB_SDONE + 2,
  FB_PVDONE = FB_PFULL + 4,
  FB_PVFREE = FB_PVDONE + 2,
  FB_ITEM = FB_PVFREE + 2,   // + item slot: the softmax wrote the item's l and m
  FB_LFREE = FB_ITEM + 2,    // + item slot: the correction's epilogue read them
  FB_DRAIN = FB_LFREE + 2,
  FB_COUNT
};
static_assert(FB_COUNT <= 32, "barriers");
// tensor-memory columns: S (FP32) [2][128], then P^ (FP16 pairs) over its
// first 64 columns; PV (FP32) [2][D]
constexpr uint32_t kTfS = 0, kTfPv = 256;

// Work item it of the forward: query tile qt of head bh, with nkt KV tiles.
// Causal items come longest first (all heads' last query tiles, then the
// tiles before them).  CTA c of G takes in round r the item r G + c (r
// even) or r G + G - 1 - c (r odd): dealt in this snake order, the causal
// items' lengths even out over the CTAs (imbalance 14% -> 2% on 16 heads of
// 64 query tiles, against dealing every round forward).
struct FwdItem {
  int qt, bh, nkt;
};
__device__ __forceinline__ int fwd_item_index(int r, int c, int G) { return r * G + ((r & 1) ? G - 1 - c : c); }
template <bool kCausal>
__device__ __forceinline__ FwdItem fwd_item(int it, int nqt, int BH) {
  FwdItem r;
  if (kCausal) {
    r.qt = nqt - 1 - it / BH;
    r.bh = it % BH;
    r.nkt = r.qt + 1;
  } else {
    r.bh = it / nqt;
    r.qt = it % nqt;
    r.nkt = nqt;
  }
  return r;
}

// Q^ or K^ rows [rows .. rows + 127] into a [D / 64][128][64] tile (halves 16
// KB apart): at D = 64 one bulk copy; at D = 128 two tiled copies of 128-byte
// column halves (the rows' 16-byte chunks are XOR-permuted within each half,
// so the copies land in the tensor core's 128-byte-swizzled layout).
template <int D>
__device__ __forceinline__ void load_rows(uint32_t dst, const uint16_t* src, const CUtensorMap* map, int row0,
                                          uint32_t bar) {
  if constexpr (D == 64) {
    bulk_load(dst, src + static_cast<size_t>(row0) * D, 128 * 128, bar);
  } else {
    sagefp4::tma_load_2d(dst, map, 0, row0, bar);
    sagefp4::tma_load_2d(dst + 128 * 128, map, 128, row0, bar);
  }
}

template <int D, bool kCausal>
__global__ void __launch_bounds__(kTcThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, Ws ws,
                  uint16_t* __restrict__ out, float* __restrict__ lse, int N, int BH, float scale_log2e,
                  uint64_t wait_ns, int withhold) {
  using L = TfSmem<D>;
  constexpr int kSt = L::kStages;
  // K^ and V^T rings refilled separately (at D = 64 together: measured 3%
  // faster, the softmax sets the pace there)
  constexpr bool kSplit = D == 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const int nqt = (N + kTok - 1) / kTok;
  const int Np = nqt * kTok;
  const int n_items = nqt * BH, cta = static_cast<int>(blockIdx.x), ncta = static_cast<int>(gridDim.x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wg = warp >> 2;
  const Ctl ctl{ws.status, wait_ns};
  auto bar = [&](int i) { return sbase + L::kBarOff + 8 * i; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  float* xm = reinterpret_cast<float*>(smem + L::kXm);     // [2 parity][2 halves][128 rows]
  float* al = reinterpret_cast<float*>(smem + L::kAl);     // [tile mod 4][128 rows]
  float* bm = reinterpret_cast<float*>(smem + L::kBm);     // [2 parity][8 softmax warps]
  float* beta = reinterpret_cast<float*>(smem + L::kBeta); // [tile mod 4][2 row blocks]
  float* lf = reinterpret_cast<float*>(smem + L::kLf);     // [2 item slots][2 halves][128 rows]
  float* mf = reinterpret_cast<float*>(smem + L::kMf);     // [2 item slots][128 rows]

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2; q++) {
      mbar_init(bar(FB_Q + q), 1);
      mbar_init(bar(FB_QEMPTY + q), 1);  // the MMA commit after the item's last S
      mbar_init(bar(FB_ITEM + q), 8);
      mbar_init(bar(FB_LFREE + q), 4);
    }
    for (int s = 0; s < kSt; s++) {
      mbar_init(bar(FB_KFULL + s), 1);
      mbar_init(bar(FB_VFULL + s), 1);
      mbar_init(bar(FB_KEMPTY + s), 1);  // the MMA commit after S
      mbar_init(bar(FB_VEMPTY + s), 1);  // the MMA commit after PV
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(bar(FB_SDONE + b), 1);
      mbar_init(bar(FB_PVDONE + b), 1);
      mbar_init(bar(FB_PVFREE + b), 4);
    }
    for (int q = 0; q < 4; q++) mbar_init(bar(FB_PFULL + q), 8);
    mbar_init(bar(FB_DRAIN), 1);
    *abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (wg == 0) {
    sagefp4::regs_dec<TcRegs::kCtl>();
    if ((warp == 0 || (kSplit && warp == 2)) && lane == 0) {
      // ---- producers: warp 0 Q^ and the K^ tiles, warp 2 the V^T tiles,
      // each ring refilled as soon as its own product has read the slot (at
      // D = 64 warp 0 copies both, and a stage is refilled after PV); a Q^
      // slot once every S of the item two before has completed
      const bool isk = warp == 0;
      const int full = isk ? FB_KFULL : FB_VFULL, empty = isk && kSplit ? FB_KEMPTY : FB_VEMPTY;
      const bool held = isk && withhold && blockIdx.x == 0;
      int g = 0, issued = 0, nq = 0;
      bool run = true;
      for (int i = 0; run; i++) {
        const int it = fwd_item_index(i, cta, ncta);
        if (it >= n_items) break;
        const FwdItem I = fwd_item<kCausal>(it, nqt, BH);
        const int hrow = I.bh * Np;  // the head's first row in [B*H*Np][D]
        const size_t hb = static_cast<size_t>(I.bh) * Np * D;
        if (isk) {
          const int qs = i & 1;
          if (i >= 2 && !wait1_ab(bar(FB_QEMPTY + qs), ((i >> 1) - 1) & 1, ctl, abort)) break;
          mbar_arrive_expect_tx(bar(FB_Q + qs), L::kQBytes);
          load_rows<D>(sbase + L::kQ + qs * L::kQBytes, ws.qc, &tm_q, hrow + I.qt * kTok, bar(FB_Q + qs));
          nq = i + 1;
        }
        for (int kt = 0; kt < I.nkt; kt++, g++) {
          const int s = g % kSt;
          if (g >= kSt && !wait1_ab(bar(empty + s), ((g / kSt) - 1) & 1, ctl, abort)) {
            run = false;
            break;
          }
          if (held && g == 0) continue;  // failure-detection test: this tile never arrives
          const uint32_t st = sbase + L::kStageOff + s * L::kStage;
          mbar_arrive_expect_tx(bar(full + s), kSplit ? L::kStage / 2 : L::kStage);
          if (isk) load_rows<D>(st + L::kSK, ws.kc, &tm_k, hrow + kt * kTok, bar(full + s));
          if (!isk || !kSplit)
            bulk_load(st + L::kSV, ws.vct + hb + static_cast<size_t>(kt) * kTok * D, L::kStage / 2, bar(full + s));
          issued = g + 1;
        }
      }
      if (*abort) {
        // let every copy this thread issued land before the CTA exits
        for (int last = issued - 1; last >= 0 && last >= issued - kSt; last--)
          if (!(held && last == 0)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar(full + last % kSt), (last / kSt) & 1) && globaltimer_ns() - t0 < ctl.limit) {
            }
          }
        for (int j = nq > 2 ? nq - 2 : 0; j < nq; j++) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar(FB_Q + (j & 1)), (j >> 1) & 1) && globaltimer_ns() - t0 < ctl.limit) {
          }
        }
      }
    } else if (warp == 1) {
      // ---- MMA issue: the whole warp, one elected lane issues.  S runs one
      // tile of the stream ahead of PV; its cursor (item, tile) crosses into
      // the next item, whose Q^ slot it waits for at the item's first tile.
      const uint32_t idS = idesc_f16(128, 128), idPV = idesc_f16(128, D);
      int total = 0;  // tiles of this CTA's stream
      for (int r = 0, it; (it = fwd_item_index(r, cta, ncta)) < n_items; r++) total += fwd_item<kCausal>(it, nqt, BH).nkt;
      int s_g = 0, s_i = 0, s_kt = 0, s_nkt = total > 0 ? fwd_item<kCausal>(cta, nqt, BH).nkt : 0;
      // descriptors: a K step of 16 moves 32 bytes (+2), a 64-wide half 16 KB
      // (+1024); V^T's key halves are D * 128 bytes apart
      auto issue_s = [&]() {
        const int g = s_g, s = g % kSt, b = g & 1, qs = s_i & 1;
        if (s_kt == 0 && !waitw_ab(bar(FB_Q + qs), (s_i >> 1) & 1, ctl, abort)) return false;
        if (!waitw_ab(bar(FB_KFULL + s), (g / kSt) & 1, ctl, abort)) return false;
        // buffer b: PV of tile g - 2 has read its P^ (and so the softmax has
        // read its S); PV's latest completion can be tile g - 2's here
        if (g >= 2 && !waitw_ab(bar(FB_PVDONE + b), ((g >> 1) - 1) & 1, ctl, abort)) return false;
        tc_fence_after();
        const uint64_t dq0 = desc_k64(sbase + L::kQ + qs * L::kQBytes, 0);
        const uint64_t dks = desc_k64(sbase + L::kStageOff + s * L::kStage + L::kSK, 0);
        const bool last = s_kt == s_nkt - 1;
        if (elect1()) {
#pragma unroll
          for (int k = 0; k < D / 16; k++)
            mma_f16_tc(tmem + kTfS + 128 * b, dq0 + 1024 * (k >> 2) + 2 * (k & 3), dks + 1024 * (k >> 2) + 2 * (k & 3),
                       idS, k > 0);
          tc_commit(bar(FB_SDONE + b));
          if constexpr (kSplit) tc_commit(bar(FB_KEMPTY + s));
          if (last) tc_commit(bar(FB_QEMPTY + qs));  // the item's Q^ slot can take item i + 2
        }
        __syncwarp();
        s_g++;
        if (last) {
          s_kt = 0;
          s_i++;
          const int nit = fwd_item_index(s_i, cta, ncta);
          s_nkt = nit < n_items ? fwd_item<kCausal>(nit, nqt, BH).nkt : 0;
        } else {
          s_kt++;
        }
        return true;
      };
      bool ok = total == 0 || issue_s();
      for (int g = 0; ok && g < total; g++) {
        const int s = g % kSt, b = g & 1;
        if (g + 1 < total && !(ok = issue_s())) break;
        if (!(ok = waitw_ab(bar(FB_PFULL + (g & 3)), (g >> 2) & 1, ctl, abort))) break;
        if (g >= 2 && !(ok = waitw_ab(bar(FB_PVFREE + b), ((g >> 1) - 1) & 1, ctl, abort))) break;
        if (kSplit && !(ok = waitw_ab(bar(FB_VFULL + s), (g / kSt) & 1, ctl, abort))) break;
        tc_fence_after();
        // A: P^ over S's first 64 columns (8 columns a K step of 16 keys)
        const uint64_t dvs = desc_k64(sbase + L::kStageOff + s * L::kStage + L::kSV, 0);
        if (elect1()) {
#pragma unroll
          for (int k = 0; k < 8; k++)
            mma_f16_tc_ta(tmem + kTfPv + D * b, tmem + kTfS + 128 * b + 8 * k, dvs + 8 * D * (k >> 2) + 2 * (k & 3),
                          idPV, k > 0);
          tc_commit(bar(FB_PVDONE + b));
          tc_commit(bar(FB_VEMPTY + s));
        }
        __syncwarp();
      }
      if (elect1()) tc_commit(bar(FB_DRAIN));
      __syncwarp();
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar(FB_DRAIN), 0) && globaltimer_ns() - t0 < ctl.limit) {
      }
    }
    // end of the CTA: every role arrives from its own code path (barrier 2)
    __syncwarp();
    named_bar(2, kTcThreads);
    if (warp == 1) tmem_dealloc(tmem, 512);
  } else if (wg == 1 || wg == 2) {
    // ---- softmax: this thread's query row, keys 64h..64h+63 of each tile.
    // The scores arrive as exact integers (Q^.K^ code products); the scale
    // sq sk scale log2(e) enters only the exponent's argument.
    sagefp4::regs_inc<TcRegs::kSoft>();
    const int h = wg - 1;
    const int wq = warp & 3;
    const int row = 32 * wq + lane;
    const int sw = 4 * h + wq;
    const int blk = wq >> 1;  // 64-row block of this row
    const uint32_t lanebase = static_cast<uint32_t>(32 * wq) << 16;
    const uint64_t magic2 = pack2(kRintMagic, kRintMagic), nmagic2 = pack2(-kRintMagic, -kRintMagic);
    bool ok = true;
    int g = 0;
    for (int i = 0; ok; i++) {
      const int it = fwd_item_index(i, cta, ncta);
      if (it >= n_items) break;
      const FwdItem I = fwd_item<kCausal>(it, nqt, BH);
      const int qt = I.qt, nkt = I.nkt;
      const size_t hs = static_cast<size_t>(I.bh) * nqt;  // the head's block scales
      const int qrow = qt * kTok + row;
      const bool valid = qrow < N;
      const float sqk = ws.sq[hs + qt] * scale_log2e;
      float m = -INFINITY, l = 0.0f;
      float sk_next = ws.sk[hs], sv_next = ws.sv[hs];
      for (int kt = 0; kt < nkt; kt++, g++) {
        const int b = g & 1;
        const float sk_cur = sk_next, sv_cur = sv_next;
        if (kt + 1 < nkt) {
          sk_next = ws.sk[hs + kt + 1];
          sv_next = ws.sv[hs + kt + 1];
        }
        ok = waitw_ab(bar(FB_SDONE + b), (g >> 1) & 1, ctl, abort);
        tc_fence_after();
        uint32_t ru[2][32];
        tmem_ld32(tmem + lanebase + kTfS + 128 * b + 64 * h, ru[0]);
        tmem_ld32(tmem + lanebase + kTfS + 128 * b + 64 * h + 32, ru[1]);
        tmem_wait_ld();
        if ((kCausal && kt == qt) || (kt == nqt - 1 && (N % kTok) != 0)) {
          // keys past N, and (causal) past this row, do not take part
          const int k0 = kt * kTok + 64 * h;
          const int lastk = kCausal ? min(N - 1, qrow) : N - 1;
#pragma unroll
          for (int e = 0; e < 64; e++)
            if (k0 + e > lastk) ru[e >> 5][e & 31] = __float_as_uint(-INFINITY);
        }
        float hm;
        {
          float t[8];
#pragma unroll
          for (int j = 0; j < 8; j++) {
            const uint32_t* r = &ru[j >> 2][(j & 3) * 8];
            t[j] = max3f(max3f(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2])),
                         max3f(__uint_as_float(r[3]), __uint_as_float(r[4]), __uint_as_float(r[5])),
                         fmaxf(__uint_as_float(r[6]), __uint_as_float(r[7])));
          }
          hm = max3f(max3f(t[0], t[1], t[2]), max3f(t[3], t[4], t[5]), fmaxf(t[6], t[7]));
        }
        // the row's maximum over both halves of the tile (xm by tile parity)
        xm[(2 * b + h) * 128 + row] = hm;
        // alpha and beta go to slot g % 4, which the correction has read for
        // tile g - 4: S of this tile was issued after PV of tile g - 2, and
        // that PV after the correction had released tile g - 4's PV buffer.
        // The vote also publishes xm, and orders both halves' loads of S
        // before P^ overwrites its first 64 columns
        if (!(ok = group_and(ok))) break;
        const float mt = fmaxf(hm, xm[(2 * b + 1 - h) * 128 + row]);
        // c2 > 0 keeps masked keys at -inf (c2 = 0 only when every score is 0)
        const float c2 = fmaxf(sqk * sk_cur, 1e-30f);
        const float mn = fmaxf(m, mt * c2);
        const float alpha = ex2(m - mn);  // m = -inf on the item's first tile: 0
        m = mn;
        // The block's largest P~ is the largest of its rows' maxima, each the
        // exponential of the same argument as the row's largest score (rows past
        // N excluded); both halves of a row compute it alike, so each half takes
        // the block maximum over its own two warps.
        const float rp = valid ? ex2(fmaf(mt, c2, -mn)) : 0.0f;
        const uint32_t wmax = redux_max_u32(__float_as_uint(rp) & 0x7fffffffu);  // rp >= 0: bit order is value order
        if (lane == 0) bm[b * 8 + sw] = __uint_as_float(wmax);
        if (h == 0) al[(g & 3) * 128 + row] = alpha;
        named_bar(3 + 2 * h + blk, 64);  // publishes bm to the block's other warp of this half
        const float amax = fmaxf(bm[b * 8 + 4 * h + 2 * blk], bm[b * 8 + 4 * h + 2 * blk + 1]);
        const float inv = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
        if (h == 0 && wq == 2 * blk && lane == 0) beta[(g & 3) * 2 + blk] = __fdiv_rn(amax, 127.0f) * sv_cur;
        // one pass: P~ = exp2(s c2 - m), its row sum, and its codes
        // rint(P~ * inv): P~ * inv + 1.5 * 2^23 in one FMA rounds the exact
        // product to an integer (ties to even), and subtracting 1.5 * 2^23 is
        // exact
        const uint64_t c22 = pack2(c2, c2), nm2 = pack2(-mn, -mn), ii = pack2(inv, inv);
        uint64_t acc0 = 0, acc1 = 0;
        uint32_t pw[32];  // keys 2j, 2j + 1 of this half as FP16 codes
#pragma unroll
        for (int j = 0; j < 32; j++) {
          const uint32_t* r = &ru[j >> 4][(j & 15) * 2];
          const uint64_t y = fma2(pack2(__uint_as_float(r[0]), __uint_as_float(r[1])), c22, nm2);
          const uint64_t x = pack2(ex2(lo2(y)), ex2(hi2(y)));
          if (j & 1)
            acc1 = add2(acc1, x);
          else
            acc0 = add2(acc0, x);
          const uint64_t n = add2(fma2(x, ii, magic2), nmagic2);
          pw[j] = h2(lo2(n), hi2(n));
        }
        const uint64_t acc = add2(acc0, acc1);
        l = fmaf(l, alpha, lo2(acc) + hi2(acc));
        tmem_st32(tmem + lanebase + kTfS + 128 * b + 32 * h, pw);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive1(bar(FB_PFULL + (g & 3)));
      }
      if (!ok) break;
      // the item's row statistics for its epilogue, in slot i % 2 once the
      // correction has read item i - 2's (voted, so that all eight warps
      // leave together if the wait runs out)
      const int ls = i & 1;
      ok = i < 2 || waitw_ab(bar(FB_LFREE + ls), ((i >> 1) - 1) & 1, ctl, abort);
      if (!(ok = group_and(ok))) break;
      lf[(2 * ls + h) * 128 + row] = l;
      if (h == 0) mf[ls * 128 + row] = m;
      __syncwarp();
      if (lane == 0) mbar_arrive1(bar(FB_ITEM + ls));
    }
    tc_fence_before();
    named_bar(2, kTcThreads);
  } else {
    // ---- correction: O of this thread's row, as FP32 pairs
    sagefp4::regs_inc<TcRegs::kFold>();
    const int row = 32 * (warp & 3) + lane;
    const int blk = (warp & 3) >> 1;
    const uint32_t lanebase = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    bool ok = true;
    int g = 0;
    for (int i = 0; ok; i++) {
      const int it = fwd_item_index(i, cta, ncta);
      if (it >= n_items) break;
      const FwdItem I = fwd_item<kCausal>(it, nqt, BH);
      uint64_t o[D / 2];
#pragma unroll
      for (int c = 0; c < D / 2; c++) o[c] = 0;
      for (int kt = 0; kt < I.nkt; kt++, g++) {
        const int b = g & 1;
        // PFULL: the softmax's alpha and beta of this tile (its release); PVDONE: the product
        if (!(ok = waitw_ab(bar(FB_PFULL + (g & 3)), (g >> 2) & 1, ctl, abort))) break;
        if (!(ok = waitw_ab(bar(FB_PVDONE + b), (g >> 1) & 1, ctl, abort))) break;
        tc_fence_after();
        const float alpha = al[(g & 3) * 128 + row], bt = beta[(g & 3) * 2 + blk];
        // o = pv * beta + o * alpha; o * 1 is o, so warps whose rows' maxima
        // all held skip the multiply
        const uint64_t bt2 = pack2(bt, bt), al2 = pack2(alpha, alpha);
        const bool keep = __all_sync(kFull, alpha == 1.0f);
#pragma unroll
        for (int c = 0; c < D / 32; c++) {
          uint32_t ru[32];
          tmem_ld32(tmem + lanebase + kTfPv + D * b + 32 * c, ru);
          tmem_wait_ld();
          if (keep) {
#pragma unroll
            for (int j = 0; j < 16; j++)
              o[16 * c + j] =
                  fma2(pack2(__uint_as_float(ru[2 * j]), __uint_as_float(ru[2 * j + 1])), bt2, o[16 * c + j]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; j++)
              o[16 * c + j] = fma2(pack2(__uint_as_float(ru[2 * j]), __uint_as_float(ru[2 * j + 1])), bt2,
                                   mul2(o[16 * c + j], al2));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive1(bar(FB_PVFREE + b));
      }
      if (!ok) break;
      // the item's epilogue, once the softmax has published its l and m
      const int ls = i & 1;
      if (!(ok = waitw_ab(bar(FB_ITEM + ls), (i >> 1) & 1, ctl, abort))) break;
      const int qrow = I.qt * kTok + row;
      if (qrow < N && !*abort) {
        const float lt = lf[2 * ls * 128 + row] + lf[(2 * ls + 1) * 128 + row];
        const float il = 1.0f / lt;
        uint16_t* orow = out + (static_cast<size_t>(I.bh) * N + qrow) * D;
#pragma unroll
        for (int c = 0; c < D / 8; c++) {
          __nv_bfloat162 h0 = __floats2bfloat162_rn(lo2(o[4 * c + 0]) * il, hi2(o[4 * c + 0]) * il);
          __nv_bfloat162 h1 = __floats2bfloat162_rn(lo2(o[4 * c + 1]) * il, hi2(o[4 * c + 1]) * il);
          __nv_bfloat162 hh2 = __floats2bfloat162_rn(lo2(o[4 * c + 2]) * il, hi2(o[4 * c + 2]) * il);
          __nv_bfloat162 h3 = __floats2bfloat162_rn(lo2(o[4 * c + 3]) * il, hi2(o[4 * c + 3]) * il);
          uint4 w;
          w.x = *reinterpret_cast<uint32_t*>(&h0);
          w.y = *reinterpret_cast<uint32_t*>(&h1);
          w.z = *reinterpret_cast<uint32_t*>(&hh2);
          w.w = *reinterpret_cast<uint32_t*>(&h3);
          *reinterpret_cast<uint4*>(orow + 8 * c) = w;
        }
        lse[static_cast<size_t>(I.bh) * N + qrow] = (mf[ls * 128 + row] + __log2f(lt)) * kLn2;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive1(bar(FB_LFREE + ls));
    }
    tc_fence_before();
    named_bar(2, kTcThreads);
  }
}

// dQ accumulator (FP32, padded rows) -> bf16 [BH][N][D]
template <int D>
__global__ void __launch_bounds__(kThreads) dq_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq, int N,
                                                      int BH) {
  const int Np = (N + kTok - 1) / kTok * kTok;
  const size_t total = static_cast<size_t>(BH) * N * D / 4;
  for (size_t i = blockIdx.x * static_cast<size_t>(kThreads) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * kThreads) {
    const size_t e = 4 * i;
    const size_t row = e / D, d = e % D;
    const size_t bh = row / N, n = row % N;
    const float4 v = *reinterpret_cast<const float4*>(acc + (bh * Np + n) * D + d);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&lo);
    w.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dq + e) = w;
  }
}

// ---------------------------------------------------------------- probes
// tcgen05 kind::f16 with the layouts the kernels use: one CTA of 4 warps
// computes C [128][N] = A [128][64] x B [N][64]^T (FP16 in, FP32 out) from
// row-major global inputs staged into swizzled shared memory.
__global__ void __launch_bounds__(128) umma_probe_kernel(const uint16_t* __restrict__ a, const uint16_t* __restrict__ b,
                                                         int N, float* __restrict__ c, int32_t* status) {
  __shared__ __align__(1024) uint8_t sa[128 * 128];
  __shared__ __align__(1024) uint8_t sb[128 * 128];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 128 * 8; i += 128) {  // 16-byte chunks of A
    const int r = i / 8, ch = i % 8;
    *reinterpret_cast<uint4*>(sa + swz(r, 16 * ch, 128)) = *reinterpret_cast<const uint4*>(a + r * 64 + 8 * ch);
  }
  for (int i = tid; i < N * 8; i += 128) {
    const int r = i / 8, ch = i % 8;
    *reinterpret_cast<uint4*>(sb + swz(r, 16 * ch, 128)) = *reinterpret_cast<const uint4*>(b + r * 64 + 8 * ch);
  }
  if (tid == 0) {
    mbar_init(smem_addr(&bar), 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(&tslot), 128);
    tmem_relinquish();
  }
  // generic-proxy writes of the operands -> visible to the tensor core
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  if (tid == 0) {
    const uint32_t id = idesc_f16(128, N);
#pragma unroll
    for (int k = 0; k < 4; k++)
      mma_f16_tc(tmem, desc_k64(smem_addr(sa), 16 * k), desc_k64(smem_addr(sb), 16 * k), id, k > 0);
    tc_commit(smem_addr(&bar));
  }
  const Ctl ctl{status, 100ull * 1000ull * 1000ull};
  const bool ok = waitw(smem_addr(&bar), 0, ctl);
  tc_fence_after();
  if (ok) {
    const int row = 32 * warp + (tid & 31);
    for (int c0 = 0; c0 < N; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; j++) c[row * N + c0 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// Probe of the MN-major form: one CTA computes c [128][64] = a [128][128] x
// b [128][64] (FP16 in, FP32 out, row-major device arrays) with both operands
// staged K-row by K-row, A's two 64-row blocks of M 32 KB apart (as dQ reads
// two query tiles' dS^ codes from two buffers) and B between them.
constexpr int kMnProbeSmem = 3 * 16384 + 1024;
__global__ void __launch_bounds__(128) umma_mn_probe_kernel(const uint16_t* __restrict__ a,
                                                            const uint16_t* __restrict__ b, float* __restrict__ c,
                                                            int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr int kA0 = 0, kB = 16384, kA1 = 32768;
  for (int i = tid; i < 128 * 128; i += 128) {  // a[m][k] -> row k of block m / 64
    const int m = i >> 7, k = i & 127;
    *reinterpret_cast<uint16_t*>(sm + (m < 64 ? kA0 : kA1) + swz(k, 2 * (m & 63), 128)) = a[i];
  }
  for (int i = tid; i < 128 * 64; i += 128) {  // b[k][n] -> row k
    const int k = i >> 6, n = i & 63;
    *reinterpret_cast<uint16_t*>(sm + kB + swz(k, 2 * n, 128)) = b[i];
  }
  if (tid == 0) {
    mbar_init(smem_addr(&bar), 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(&tslot), 64);
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  const uint32_t sb = smem_addr(sm);
  if (tid == 0) {
    const uint32_t id = idesc_f16_mn(128, 64);
#pragma unroll
    for (int k = 0; k < 8; k++)
      mma_f16_tc(tmem, desc_mn(sb + kA0, 16 * k, kA1 - kA0), desc_mn(sb + kB, 16 * k, kA1 - kA0), id, k > 0);
    tc_commit(smem_addr(&bar));
  }
  const Ctl ctl{status, 100ull * 1000ull * 1000ull};
  const bool ok = waitw(smem_addr(&bar), 0, ctl);
  tc_fence_after();
  if (ok) {
    const int row = 32 * warp + (tid & 31);
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; j++) c[row * 64 + c0 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}


// Integer products on the FP16 MMA: one warp computes the 16 x 8 product of
// INT8 matrices a [16][K] and b [8][K] (both row-major, K a multiple of 16)
// with the codes as FP16 values and FP32 accumulation, chained over K / 16
// MMAs like the kernels' sums, and writes it as float [16][8].
__global__ void int_mma_probe_kernel(const int8_t* __restrict__ a, const int8_t* __restrict__ b, int K,
                                     float* __restrict__ out) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  for (int ks = 0; ks < K / 16; ks++) {
    const int k0 = 16 * ks + 2 * t;
    uint32_t fa[4];
    fa[0] = h2(a[g * K + k0], a[g * K + k0 + 1]);
    fa[1] = h2(a[(g + 8) * K + k0], a[(g + 8) * K + k0 + 1]);
    fa[2] = h2(a[g * K + k0 + 8], a[g * K + k0 + 9]);
    fa[3] = h2(a[(g + 8) * K + k0 + 8], a[(g + 8) * K + k0 + 9]);
    const uint32_t b0 = h2(b[g * K + k0], b[g * K + k0 + 1]);
    const uint32_t b1 = h2(b[g * K + k0 + 8], b[g * K + k0 + 9]);
    mma_f16(c, fa, b0, b1);
  }
  out[g * 8 + 2 * t] = c[0];
  out[g * 8 + 2 * t + 1] = c[1];
  out[(g + 8) * 8 + 2 * t] = c[2];
  out[(g + 8) * 8 + 2 * t + 1] = c[3];
}

// Throughput of the warp-level MMA forms on register operands: kind 0 INT8
// m16n8k32, kind 1 FP16 m16n8k16 with FP32 accumulation (the one the kernels
// use).  Eight independent accumulators per warp.
template <int kKind>
__global__ void __launch_bounds__(kThreads) mma_peak_kernel(int iters, int* out) {
  uint32_t a[4], b0, b1;
  const uint32_t seed = threadIdx.x * 0x9E3779B9u + blockIdx.x;
  a[0] = seed;
  a[1] = seed ^ 0x5bd1e995u;
  a[2] = seed * 3u;
  a[3] = seed + 0x1234567u;
  b0 = seed ^ 0xabcdefu;
  b1 = seed * 7u;
  if (kKind == 0) {
    int c[8][4] = {};
    for (int i = 0; i < iters; i++)
#pragma unroll
      for (int u = 0; u < 8; u++) mma_s8(c[u], a, b0, b1);
    int s = 0;
#pragma unroll
    for (int u = 0; u < 8; u++) s += c[u][0] + c[u][1] + c[u][2] + c[u][3];
    if (s == 0x7fffffff) out[0] = s;
  } else {
    // small FP16 values so the sums stay finite
    a[0] = a[1] = a[2] = a[3] = 0x3c003c00u & (seed | 0x3c003c00u);
    b0 = b1 = 0x1c001c00u;
    float c[8][4] = {};
    for (int i = 0; i < iters; i++)
#pragma unroll
      for (int u = 0; u < 8; u++) mma_f16(c[u], a, b0, b1);
    float s = 0.0f;
#pragma unroll
    for (int u = 0; u < 8; u++) s += c[u][0] + c[u][1] + c[u][2] + c[u][3];
    if (s == -1.0f) out[0] = 1;
  }
}

// Throughput of the 5th-generation forms the kernels use (tcgen05.mma
// kind::f16, M = 128, K = 16, N = kN): one thread per CTA issues iters x 8
// MMAs back to back into one tensor-memory accumulator from zero-filled
// 128-byte-swizzled operands, then waits (bounded) for their completion; a
// wait that runs out writes SAGE_FP4_ETIMEOUT to out[0].  kForm 0: A and B
// K-major in shared memory; 1: A in tensor memory; 2: B MN-major.
template <int kN, int kForm>
__global__ void __launch_bounds__(128, 1) umma_peak_kernel(int iters, int* out) {
  // A (128 rows) and B (kN rows) share one zero-filled buffer
  __shared__ __align__(1024) uint8_t sb[(kN > 128 ? kN : 128) * 128];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  uint8_t* sa = sb;
  for (int i = tid; i < (kN > 128 ? kN : 128) * 8; i += 128) reinterpret_cast<uint4*>(sb)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    mbar_init(smem_addr(&bar), 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(&tslot), 256);
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  if (tid == 0) {
    const uint32_t id = kForm == 2 ? (idesc_f16(128, kN) | (1u << 16)) : idesc_f16(128, kN);
    const uint64_t da = desc_k64(smem_addr(sa), 0);
    const uint64_t db = kForm == 2 ? desc_mn(smem_addr(sb), 0, 8192) : desc_k64(smem_addr(sb), 0);
    for (int i = 0; i < iters; i++)
#pragma unroll
      for (int k = 0; k < 8; k++) {
        if (kForm == 1)
          mma_f16_tc_ta(tmem, tmem + 128 + 8 * (k & 3), db + 2 * (k & 3), id, (i | k) != 0);
        else if (kForm == 2)
          mma_f16_tc(tmem, da + 2 * (k & 3), db + 128 * (k & 3), id, (i | k) != 0);
        else
          mma_f16_tc(tmem, da + 2 * (k & 3), db + 2 * (k & 3), id, (i | k) != 0);
      }
    tc_commit(smem_addr(&bar));
    const uint64_t t0 = globaltimer_ns();
    bool done = false;
    while (!(done = mbar_try_wait(smem_addr(&bar), 0)) && globaltimer_ns() - t0 < 1000000000ull) {
    }
    if (!done) out[0] = SAGE_FP4_ETIMEOUT;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// Probe of the A-in-tensor-memory form: one CTA computes c [128][N] =
// a [128][64] x b [N][64]^T (FP16 in, FP32 out, row-major device arrays) with
// A written to tensor memory by tcgen05.st (thread = row) and B in shared
// memory (128-byte-swizzled K-major).
__global__ void __launch_bounds__(128) umma_ta_probe_kernel(const uint16_t* __restrict__ a,
                                                            const uint16_t* __restrict__ b, int N,
                                                            float* __restrict__ c, int32_t* status) {
  __shared__ __align__(1024) uint8_t sb[128 * 128];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < N * 8; i += 128) {
    const int r = i / 8, ch = i % 8;
    *reinterpret_cast<uint4*>(sb + swz(r, 16 * ch, 128)) = *reinterpret_cast<const uint4*>(b + r * 64 + 8 * ch);
  }
  if (tid == 0) {
    mbar_init(smem_addr(&bar), 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(&tslot), 256);
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  const uint32_t lanebase = static_cast<uint32_t>(32 * warp) << 16;
  {
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; j++)
      r[j] = static_cast<uint32_t>(a[tid * 64 + 2 * j]) | (static_cast<uint32_t>(a[tid * 64 + 2 * j + 1]) << 16);
    tmem_st32(tmem + lanebase + 128, r);  // A in columns 128..159
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t id = idesc_f16(128, N);
    const uint64_t db = desc_k64(smem_addr(sb), 0);
#pragma unroll
    for (int k = 0; k < 4; k++) mma_f16_tc_ta(tmem, tmem + 128 + 8 * k, db + 2 * k, id, k > 0);
    tc_commit(smem_addr(&bar));
  }
  const Ctl ctl{status, 100ull * 1000ull * 1000ull};
  const bool ok = waitw(smem_addr(&bar), 0, ctl);
  tc_fence_after();
  if (ok) {
    const int row = 32 * warp + (tid & 31);
    for (int c0 = 0; c0 < N; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lanebase + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; j++) c[row * N + c0 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------- host side
struct Layout {
  size_t off[SAGEBWD_WS_FIELDS];
  size_t total;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

Layout layout(int B, int H, int N, int D) {
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t Np = (static_cast<size_t>(N) + kTok - 1) / kTok * kTok;
  const size_t nb = Np / kTok;
  const size_t rows = 2 * BH * Np * D;  // FP16 [BH][Np][D]
  const size_t sizes[SAGEBWD_WS_FIELDS] = {
      rows,        rows,        rows,        rows,         // Q^, K^, V^, dO^ codes
      rows,        rows,                                   // V, dO as FP16
      rows,        rows,                                   // Q^, dO^ codes transposed per 64-token tile
      rows,                                                // V^ codes transposed per 64-token half tile
      4 * BH * nb, 4 * BH * nb, 4 * BH * nb, 4 * BH * nb,  // Q, K, V, dO block scales
      4 * BH * Np, 4 * BH * Np,                            // L (log2 units), D = rowsum(dO o O)
      4 * BH * Np * D,                                     // dQ accumulator
      256,                                                 // status word
  };
  Layout l;
  size_t off = 0;
  for (int i = 0; i < SAGEBWD_WS_FIELDS; i++) {
    l.off[i] = off;
    off += align256(sizes[i]);
  }
  l.total = off;
  return l;
}

Ws carve(void* base, const Layout& l) {
  char* b = static_cast<char*>(base);
  Ws w;
  w.qc = reinterpret_cast<uint16_t*>(b + l.off[0]);
  w.kc = reinterpret_cast<uint16_t*>(b + l.off[1]);
  w.vc = reinterpret_cast<uint16_t*>(b + l.off[2]);
  w.doc = reinterpret_cast<uint16_t*>(b + l.off[3]);
  w.vh = reinterpret_cast<uint16_t*>(b + l.off[4]);
  w.doh = reinterpret_cast<uint16_t*>(b + l.off[5]);
  w.qct = reinterpret_cast<uint16_t*>(b + l.off[6]);
  w.doct = reinterpret_cast<uint16_t*>(b + l.off[7]);
  w.vct = reinterpret_cast<uint16_t*>(b + l.off[8]);
  w.sq = reinterpret_cast<float*>(b + l.off[9]);
  w.sk = reinterpret_cast<float*>(b + l.off[10]);
  w.sv = reinterpret_cast<float*>(b + l.off[11]);
  w.sdo = reinterpret_cast<float*>(b + l.off[12]);
  w.l2 = reinterpret_cast<float*>(b + l.off[13]);
  w.dd = reinterpret_cast<float*>(b + l.off[14]);
  w.dqacc = reinterpret_cast<float*>(b + l.off[15]);
  w.status = reinterpret_cast<int32_t*>(b + l.off[16]);
  return w;
}

bool dims_ok(int B, int H, int N, int D) {
  if (B < 0 || H < 0 || N < 0 || (D != 64 && D != 128)) return false;
  const long long BH = static_cast<long long>(B) * H;
  const long long Np = (static_cast<long long>(N) + kTok - 1) / kTok * kTok;
  if (BH > 65535) return false;                 // gridDim.y
  if (Np / kTok > (1LL << 20)) return false;    // gridDim.x, with room
  if (BH * Np * D > (1LL << 40)) return false;  // workspace offsets stay sane
  return true;
}

bool aligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool scale_ok(float s) { return s > 0.0f && s < 1e30f; }  // false for NaN

int check_device() {
  static int cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SAGE_FP4_ECUDA;
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev] == 1 ? SAGE_FP4_OK : SAGE_FP4_EUNSUPPORTED;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return SAGE_FP4_ECUDA;
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) cache[dev] = ok ? 1 : 2;
  return ok ? SAGE_FP4_OK : SAGE_FP4_EUNSUPPORTED;
}

// The tcgen05 backward (D = 64).  Its warpgroups' setmaxnreg budgets add up
// to exactly 128 registers per thread at launch; with any other allocation
// an increase would never be granted, so it refuses to launch.
// 2-D FP32 tensor [rows][inner] (row pitch inner * 4 bytes) with boxes of
// [box_rows][box_inner], 128-byte swizzled (box_inner * 4 <= 128).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!enc) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return enc;
}

bool make_map_f32(CUtensorMap* m, const float* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                  uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte tensor [rows][inner] (row pitch inner bytes) with boxes of
// [box_rows][box_inner], copied as they are (no swizzle).
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                 uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool C>
cudaError_t launch_dkdv_tc(const Ws& w, uint16_t* dk, uint16_t* dv, int BH, int N, float scale, cudaStream_t st,
                           uint64_t wait_ns, int withhold) {
  const uint64_t rows = static_cast<uint64_t>(BH) * ((N + kTok - 1) / kTok * kTok);
  BwdMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (rows > 0x7fffffffu || !make_map_f32(&maps.dq, w.dqacc, D, rows, 32, 32)) return cudaErrorInvalidValue;
  if (D == 128 && (!make_map_u8(&maps.k, w.kc, 2 * D, rows, 128, 128) || !make_map_u8(&maps.v, w.vh, 2 * D, rows, 128, 128) ||
                   !make_map_u8(&maps.q, w.qc, 2 * D, rows, 128, 64) || !make_map_u8(&maps.doh, w.doh, 2 * D, rows, 128, 64) ||
                   !make_map_u8(&maps.doc, w.doc, 2 * D, rows, 128, 64)))
    return cudaErrorInvalidValue;
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, dkdv_tc_kernel<D, C>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != 65536 / kTcThreads) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(dkdv_tc_kernel<D, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem<D>::kAlloc);
  if (e != cudaSuccess) return e;
  // at D = 128 two CTAs per key tile, one per 64-column half of dV, dK, dQ
  const dim3 grid((N + kTok - 1) / kTok, BH, D / 64);
  dkdv_tc_kernel<D, C><<<grid, kTcThreads, TcSmem<D>::kAlloc, st>>>(maps, w, dk, dv, N, scale, wait_ns, withhold);
  return cudaGetLastError();
}

template <int D, bool C>
cudaError_t launch_fwd_tc(const Ws& w, uint16_t* o, float* lse, int BH, int N, float scale, cudaStream_t st,
                          uint64_t wait_ns, int withhold) {
  // D = 128: Q^ and K^ through tensor maps over the code arrays viewed as
  // bytes [B*H*Np][256], boxes of 128 rows x 128 bytes (no swizzle: the rows
  // carry it); D = 64 copies whole tiles and passes the maps unused
  CUtensorMap tq, tk;
  memset(&tq, 0, sizeof(tq));
  memset(&tk, 0, sizeof(tk));
  if (D == 128) {
    const uint64_t rows = static_cast<uint64_t>(BH) * ((N + kTok - 1) / kTok * kTok);
    if (rows > 0x7fffffffu || !make_map_u8(&tq, w.qc, 2 * D, rows, 128, 128) ||
        !make_map_u8(&tk, w.kc, 2 * D, rows, 128, 128))
      return cudaErrorInvalidValue;
  }
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, fwd_tc_kernel<D, C>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != 65536 / kTcThreads) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(fwd_tc_kernel<D, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, TfSmem<D>::kAlloc);
  if (e != cudaSuccess) return e;
  // persistent CTAs, one per SM at most, walking the work items
  const long long items = static_cast<long long>((N + kTok - 1) / kTok) * BH;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  fwd_tc_kernel<D, C><<<grid, kTcThreads, TfSmem<D>::kAlloc, st>>>(tq, tk, w, o, lse, N, BH, scale * kLog2e,
                                                                  wait_ns, withhold);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_quant(const Ws& w, const void* a, const void* b, const void* c, const void* o, const float* lse,
                         int BH, int N, int kind0, int nkinds, cudaStream_t st) {
  const dim3 grid((N + kTok - 1) / kTok, BH, nkinds);
  quant_kernel<D><<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(a), static_cast<const uint16_t*>(b),
                                             static_cast<const uint16_t*>(c), static_cast<const uint16_t*>(o), lse, N,
                                             kind0, w);
  return cudaGetLastError();
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? SAGE_FP4_OK : SAGE_FP4_ECUDA; }

}  // namespace sagebwd

using namespace sagebwd;

extern "C" {

size_t sagebwd_workspace_bytes(int B, int H, int N, int D) {
  if (!dims_ok(B, H, N, D)) return 0;
  return layout(B, H, N, D).total;
}

int sagebwd_workspace_layout(int B, int H, int N, int D, size_t* offsets) {
  if (!dims_ok(B, H, N, D) || !offsets) return SAGE_FP4_EINVAL;
  const Layout l = layout(B, H, N, D);
  for (int i = 0; i < SAGEBWD_WS_FIELDS; i++) offsets[i] = l.off[i];
  return SAGE_FP4_OK;
}

// Common checks of the step calls: sizes, causal flag, scale, workspace.
// Returns SAGE_FP4_OK (carry on), a negative code, or 1 for an empty problem.
static int check_common(int B, int H, int N, int D, int causal, float scale, const void* workspace,
                        size_t workspace_bytes, Layout* l) {
  if (!dims_ok(B, H, N, D) || (causal != 0 && causal != 1) || !scale_ok(scale)) return SAGE_FP4_EINVAL;
  if (!aligned(workspace, 256)) return SAGE_FP4_EINVAL;
  *l = layout(B, H, N, D);
  if (workspace_bytes < l->total) return SAGE_FP4_EINVAL;
  if (static_cast<long long>(B) * H * N == 0) return 1;
  return SAGE_FP4_OK;
}

int sagebwd_quantize_qkv(const void* q, const void* k, const void* v, int B, int H, int N, int D, void* workspace,
                         size_t workspace_bytes, void* stream) {
  Layout l;
  int rc = check_common(B, H, N, D, 0, 1.0f, workspace, workspace_bytes, &l);
  if (rc != SAGE_FP4_OK) return rc == 1 ? SAGE_FP4_OK : rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return SAGE_FP4_EINVAL;
  if ((rc = check_device()) != SAGE_FP4_OK) return rc;
  const Ws w = carve(workspace, l);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return from_cuda(D == 64 ? launch_quant<64>(w, q, k, v, nullptr, nullptr, B * H, N, 0, 3, st)
                           : launch_quant<128>(w, q, k, v, nullptr, nullptr, B * H, N, 0, 3, st));
}

int sagebwd_attn_fwd(void* o, float* lse, int B, int H, int N, int D, int causal, float scale, void* workspace,
                     size_t workspace_bytes, void* stream) {
  Layout l;
  int rc = check_common(B, H, N, D, causal, scale, workspace, workspace_bytes, &l);
  if (rc != SAGE_FP4_OK) return rc == 1 ? SAGE_FP4_OK : rc;
  if (!aligned(o, 16) || !aligned(lse, 4)) return SAGE_FP4_EINVAL;
  if ((rc = check_device()) != SAGE_FP4_OK) return rc;
  const Ws w = carve(workspace, l);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t* ob = static_cast<uint16_t*>(o);
  const int BH = B * H;
  cudaError_t e;
  if (D == 64)
    e = causal ? launch_fwd_tc<64, true>(w, ob, lse, BH, N, scale, st, kWaitNs, 0)
               : launch_fwd_tc<64, false>(w, ob, lse, BH, N, scale, st, kWaitNs, 0);
  else
    e = causal ? launch_fwd_tc<128, true>(w, ob, lse, BH, N, scale, st, kWaitNs, 0)
               : launch_fwd_tc<128, false>(w, ob, lse, BH, N, scale, st, kWaitNs, 0);
  return from_cuda(e);
}

int sagebwd_bwd_prep(const void* dout, const void* o, const float* lse, int B, int H, int N, int D, void* workspace,
                     size_t workspace_bytes, void* stream) {
  Layout l;
  int rc = check_common(B, H, N, D, 0, 1.0f, workspace, workspace_bytes, &l);
  if (rc != SAGE_FP4_OK) return rc == 1 ? SAGE_FP4_OK : rc;
  if (!aligned(dout, 16) || !aligned(o, 16) || !aligned(lse, 4)) return SAGE_FP4_EINVAL;
  if ((rc = check_device()) != SAGE_FP4_OK) return rc;
  const Ws w = carve(workspace, l);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return from_cuda(D == 64 ? launch_quant<64>(w, dout, nullptr, nullptr, o, lse, B * H, N, 3, 1, st)
                           : launch_quant<128>(w, dout, nullptr, nullptr, o, lse, B * H, N, 3, 1, st));
}

int sagebwd_attn_bwd(void* dk, void* dv, int B, int H, int N, int D, int causal, float scale, void* workspace,
                     size_t workspace_bytes, void* stream) {
  Layout l;
  int rc = check_common(B, H, N, D, causal, scale, workspace, workspace_bytes, &l);
  if (rc != SAGE_FP4_OK) return rc == 1 ? SAGE_FP4_OK : rc;
  if (!aligned(dk, 16) || !aligned(dv, 16)) return SAGE_FP4_EINVAL;
  if ((rc = check_device()) != SAGE_FP4_OK) return rc;
  const Ws w = carve(workspace, l);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t *dkb = static_cast<uint16_t*>(dk), *dvb = static_cast<uint16_t*>(dv);
  const int BH = B * H;
  cudaError_t e;
  if (D == 64)
    e = causal ? launch_dkdv_tc<64, true>(w, dkb, dvb, BH, N, scale, st, kWaitNs, 0)
               : launch_dkdv_tc<64, false>(w, dkb, dvb, BH, N, scale, st, kWaitNs, 0);
  else
    e = causal ? launch_dkdv_tc<128, true>(w, dkb, dvb, BH, N, scale, st, kWaitNs, 0)
               : launch_dkdv_tc<128, false>(w, dkb, dvb, BH, N, scale, st, kWaitNs, 0);
  return from_cuda(e);
}

int sagebwd_dq_out(void* dq, int B, int H, int N, int D, void* workspace, size_t workspace_bytes, void* stream) {
  Layout l;
  int rc = check_common(B, H, N, D, 0, 1.0f, workspace, workspace_bytes, &l);
  if (rc != SAGE_FP4_OK) return rc == 1 ? SAGE_FP4_OK : rc;
  if (!aligned(dq, 16)) return SAGE_FP4_EINVAL;
  if ((rc = check_device()) != SAGE_FP4_OK) return rc;
  const Ws w = carve(workspace, l);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  const size_t total = static_cast<size_t>(BH) * N * D / 4;
  const size_t want = (total + kThreads - 1) / kThreads;
  const int blocks = static_cast<int>(want < 152 * 16 ? want : 152 * 16);
  if (D == 64)
    dq_kernel<64><<<blocks, kThreads, 0, st>>>(w.dqacc, static_cast<uint16_t*>(dq), N, BH);
  else
    dq_kernel<128><<<blocks, kThreads, 0, st>>>(w.dqacc, static_cast<uint16_t*>(dq), N, BH);
  return from_cuda(cudaGetLastError());
}

int sagebwd_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
                int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  // every argument checked before the first launch
  Layout l;
  int rc = check_common(B, H, N, D, causal, scale, workspace, workspace_bytes, &l);
  if (rc != SAGE_FP4_OK) return rc == 1 ? SAGE_FP4_OK : rc;
  if (!aligned(o, 16) || !aligned(lse, 4)) return SAGE_FP4_EINVAL;
  rc = sagebwd_quantize_qkv(q, k, v, B, H, N, D, workspace, workspace_bytes, stream);
  if (rc != SAGE_FP4_OK) return rc;
  return sagebwd_attn_fwd(o, lse, B, H, N, D, causal, scale, workspace, workspace_bytes, stream);
}

int sagebwd_bwd(const void* dout, const void* o, const float* lse, void* dq, void* dk, void* dv, int B, int H, int N,
                int D, int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  Layout l;
  int rc = check_common(B, H, N, D, causal, scale, workspace, workspace_bytes, &l);
  if (rc != SAGE_FP4_OK) return rc == 1 ? SAGE_FP4_OK : rc;
  if (!aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16)) return SAGE_FP4_EINVAL;
  rc = sagebwd_bwd_prep(dout, o, lse, B, H, N, D, workspace, workspace_bytes, stream);
  if (rc != SAGE_FP4_OK) return rc;
  rc = sagebwd_attn_bwd(dk, dv, B, H, N, D, causal, scale, workspace, workspace_bytes, stream);
  if (rc != SAGE_FP4_OK) return rc;
  return sagebwd_dq_out(dq, B, H, N, D, workspace, workspace_bytes, stream);
}

int sagebwd_get_status(void* workspace, int B, int H, int N, int D, void* stream) {
  if (!dims_ok(B, H, N, D) || !aligned(workspace, 256)) return SAGE_FP4_EINVAL;
  const Layout l = layout(B, H, N, D);
  int32_t* status = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + l.off[SAGEBWD_WS_FIELDS - 1]);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SAGE_FP4_ECUDA;
  int32_t h = 0;
  if (cudaMemcpy(&h, status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return SAGE_FP4_ECUDA;
  if (h != 0 && cudaMemset(status, 0, sizeof(h)) != cudaSuccess) return SAGE_FP4_ECUDA;
  return h;
}

int sagebwd_stall_test(int kernel, void* out0, void* out1, int B, int H, int N, int D, float scale,
                       uint64_t wait_limit_ns, void* workspace, size_t workspace_bytes, void* stream) {
  Layout l;
  int rc = check_common(B, H, N, D, 0, scale, workspace, workspace_bytes, &l);
  if (rc != SAGE_FP4_OK) return rc == 1 ? SAGE_FP4_EINVAL : rc;
  if ((kernel != 0 && kernel != 1) || wait_limit_ns < 1000000ull || wait_limit_ns > kWaitNs) return SAGE_FP4_EINVAL;
  if (!aligned(out0, 16) || !aligned(out1, kernel == 0 ? 4 : 16)) return SAGE_FP4_EINVAL;
  if ((rc = check_device()) != SAGE_FP4_OK) return rc;
  const Ws w = carve(workspace, l);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  cudaError_t e;
  if (kernel == 0) {
    uint16_t* o = static_cast<uint16_t*>(out0);
    float* lse = static_cast<float*>(out1);
    e = D == 64 ? launch_fwd_tc<64, false>(w, o, lse, BH, N, scale, st, wait_limit_ns, 1)
                : launch_fwd_tc<128, false>(w, o, lse, BH, N, scale, st, wait_limit_ns, 1);
  } else {
    uint16_t *dkb = static_cast<uint16_t*>(out0), *dvb = static_cast<uint16_t*>(out1);
    e = D == 64 ? launch_dkdv_tc<64, false>(w, dkb, dvb, BH, N, scale, st, wait_limit_ns, 1)
                : launch_dkdv_tc<128, false>(w, dkb, dvb, BH, N, scale, st, wait_limit_ns, 1);
  }
  return from_cuda(e);
}

int sagebwd_umma_probe(const uint16_t* a, const uint16_t* b, int N, float* c, int32_t* status, void* stream) {
  if ((N != 64 && N != 128) || !aligned(a, 16) || !aligned(b, 16) || !aligned(c, 4) || !aligned(status, 4))
    return SAGE_FP4_EINVAL;
  const int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  umma_probe_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(a, b, N, c, status);
  return from_cuda(cudaGetLastError());
}

int sagebwd_umma_ta_probe(const uint16_t* a, const uint16_t* b, int N, float* c, int32_t* status, void* stream) {
  if ((N != 64 && N != 128) || !aligned(a, 2) || !aligned(b, 16) || !aligned(c, 4) || !aligned(status, 4))
    return SAGE_FP4_EINVAL;
  const int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  umma_ta_probe_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(a, b, N, c, status);
  return from_cuda(cudaGetLastError());
}

int sagebwd_umma_mn_probe(const uint16_t* a, const uint16_t* b, float* c, int32_t* status, void* stream) {
  if (!aligned(a, 2) || !aligned(b, 2) || !aligned(c, 4) || !aligned(status, 4)) return SAGE_FP4_EINVAL;
  const int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  cudaError_t e = cudaFuncSetAttribute(sagebwd::umma_mn_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       sagebwd::kMnProbeSmem);
  if (e != cudaSuccess) return from_cuda(e);
  sagebwd::umma_mn_probe_kernel<<<1, 128, sagebwd::kMnProbeSmem, static_cast<cudaStream_t>(stream)>>>(a, b, c, status);
  return from_cuda(cudaGetLastError());
}

int sagebwd_int_mma_probe(const int8_t* a, const int8_t* b, int K, float* out, void* stream) {
  if (K < 16 || K > 4096 || K % 16 != 0 || !aligned(a, 4) || !aligned(b, 4) || !aligned(out, 4))
    return SAGE_FP4_EINVAL;
  const int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  int_mma_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(a, b, K, out);
  return from_cuda(cudaGetLastError());
}

int sagebwd_mma_peak(int kind, int ctas, int iters, void* scratch, void* stream) {
  if (kind < 0 || kind > 6 || ctas < 1 || ctas > 65535 || iters < 1 || iters > (1 << 20) || !aligned(scratch, 4))
    return SAGE_FP4_EINVAL;
  const int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* out = static_cast<int*>(scratch);
  switch (kind) {
    case 0: mma_peak_kernel<0><<<ctas, kThreads, 0, st>>>(iters, out); break;
    case 1: mma_peak_kernel<1><<<ctas, kThreads, 0, st>>>(iters, out); break;
    case 2: umma_peak_kernel<64, 0><<<ctas, 128, 0, st>>>(iters, out); break;
    case 3: umma_peak_kernel<128, 0><<<ctas, 128, 0, st>>>(iters, out); break;
    case 4: umma_peak_kernel<256, 0><<<ctas, 128, 0, st>>>(iters, out); break;
    case 5: umma_peak_kernel<64, 1><<<ctas, 128, 0, st>>>(iters, out); break;
    default: umma_peak_kernel<64, 2><<<ctas, 128, 0, st>>>(iters, out); break;
  }
  return from_cuda(cudaGetLastError());
}

}  // extern "C"

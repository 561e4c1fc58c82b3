// noalloc.cu -- one-call NVFP4 attention for callers that cannot allocate
// device memory.
//
// Some callers have no way to call cudaMalloc: code that runs inside another
// framework's operator with no access to its allocator, plugins whose host
// application owns every device allocation, or code that must not allocate
// after start-up.  sage_fp4_attention_noalloc lets them run the whole path
// (quantize Q, K, V, then the fused FP4 attention) with only the buffers they
// already own: bf16 q, k, v in, bf16 o out, and an int32 status word.  The
// quantized operands, which the two-call API keeps in a caller-allocated
// workspace, live here in a fixed file-scope device array instead.
//
// That array is reserved on every GPU that loads this module and is held
// until the process exits.  Every call uses the same array: calls whose work
// overlaps on the GPU (different streams, or different host threads, without
// ordering between them) race on it and give undefined results.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>

#include "../../include/sage_fp4.h"
#include "kernels.h"
#include "layout.cuh"

using namespace sagefp4;

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // SAGE_FP4_NOALLOC_SCRATCH_BYTES

// Quantized Q, K, V^T of the current call.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

static_assert(kScratchBytes == SAGE_FP4_NOALLOC_SCRATCH_BYTES, "header and array size disagree");

struct Parts {
  size_t qc, qs, kc, ks, vc, vs, total;
};

bool dims_ok(int B, int H, int N, int D) {
  if (B < 0 || H < 0 || N < 0) return false;
  if (D != 64 && D != 128) return false;
  const long long BH = static_cast<long long>(B) * H;
  const long long Np = (static_cast<long long>(N) + 127) / 128 * 128;
  if (Np > (1LL << 30)) return false;
  if (BH * Np > INT_MAX) return false;
  return true;
}

Parts parts(int B, int H, int N, int D) {
  const size_t BH = static_cast<size_t>(B) * H;
  const OperandSizes os = operand_sizes(N, D);
  Parts p;
  size_t off = 0;
  p.qc = off;
  off += align256(BH * os.q_codes);
  p.qs = off;
  off += align256(BH * os.q_scales);
  p.kc = off;
  off += align256(BH * os.q_codes);
  p.ks = off;
  off += align256(BH * os.q_scales);
  p.vc = off;
  off += align256(BH * os.vt_codes);
  p.vs = off;
  off += align256(BH * os.vt_scales);
  p.total = off;
  return p;
}

bool aligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device address of g_scratch, looked up once per device with that device
// current.  In host code g_scratch names a host-side stand-in, not device
// memory, so kernels must be given this address instead.
uint8_t* scratch_address(int dev) {
  static uint8_t* addr[64];
  if (dev < 0 || dev >= 64) return nullptr;
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint8_t*>(p);
  }
  return addr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool byte_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
              uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int sage_fp4_attention_noalloc(const void* q, const void* k, const void* v, void* o,
                                          int32_t* status, int B, int H, int N, int D, int causal,
                                          void* stream) {
  if (!dims_ok(B, H, N, D) || (causal != 0 && causal != 1)) return SAGE_FP4_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(status, 4))
    return SAGE_FP4_EINVAL;
  const Parts pt = parts(B, H, N, D);
  if (pt.total > kScratchBytes) return SAGE_FP4_ETOOLARGE;
  if (static_cast<long long>(B) * H * N == 0) return SAGE_FP4_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SAGE_FP4_ECUDA;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return SAGE_FP4_EUNSUPPORTED;
  uint8_t* base = scratch_address(dev);
  if (!base) return SAGE_FP4_ECUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  const int Np = round_up_int(N, 128);
  // Every byte of the quantized operands, padding included, is rewritten by
  // the quantize kernels, so nothing left by an earlier call is read.
  const Strides dense = contiguous_bhnd(H, N, D);
  if (launch_quant_rows(q, k, dense, dense, base + pt.qc, base + pt.qs, base + pt.kc, base + pt.ks, H,
                        BH, N, D, false, st) != cudaSuccess ||
      launch_quant_v(v, dense, base + pt.vc, base + pt.vs, H, BH, N, D, false, status, st) != cudaSuccess)
    return SAGE_FP4_ECUDA;
  CUtensorMap tq, tk, tv;
  const CUtensorMapSwizzle qk_swz = (D == 128) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  if (!byte_map(&tq, base + pt.qc, D / 2, static_cast<uint64_t>(BH) * Np, D / 2, 128, qk_swz) ||
      !byte_map(&tk, base + pt.kc, D / 2, static_cast<uint64_t>(BH) * Np, D / 2, 128, qk_swz) ||
      !byte_map(&tv, base + pt.vc, Np / 2, static_cast<uint64_t>(BH) * D, 64, D,
                CU_TENSOR_MAP_SWIZZLE_64B))
    return SAGE_FP4_ECUDA;
  AttnParams p;
  p.sfq = base + pt.qs;
  p.sfk = base + pt.ks;
  p.sfv = base + pt.vs;
  p.o = o;
  p.os = dense;
  p.status = status;
  p.H = H;
  p.BH = BH;
  p.N = N;
  p.Np = Np;
  p.causal = causal;
  p.n_qt = Np / 128;
  p.a = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(D)));
  p.mx = 0;
  p.flags = 0;
  p.wait_ns = kAttnWaitNs;
  return launch_attn(tq, tk, tv, p, D, st) == cudaSuccess ? SAGE_FP4_OK : SAGE_FP4_ECUDA;
}

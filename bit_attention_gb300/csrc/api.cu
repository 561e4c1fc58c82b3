// api.cu -- the C ABI declared in include/sage_fp4.h: argument checks (before
// anything touches the device), tensor-map encoding, launches, status words.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <string.h>

#include "../../include/sage_fp4.h"
#include "kernels.h"
#include "layout.cuh"

using namespace sagefp4;

namespace {

bool dims_ok(int B, int H, int N, int D) {
  if (B < 0 || H < 0 || N < 0) return false;
  if (D != 64 && D != 128) return false;
  const long long BH = static_cast<long long>(B) * H;
  const long long Np = (static_cast<long long>(N) + 127) / 128 * 128;
  if (Np > (1LL << 30)) return false;
  if (BH * Np > INT_MAX) return false;            // code rows are indexed with 32-bit ints
  if (BH * Np / 128 > static_cast<long long>(UINT_MAX)) return false;
  return true;
}

bool is_empty(int B, int H, int N) { return static_cast<long long>(B) * H * N == 0; }

bool aligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct WsLayout {
  size_t qc, qs, kc, ks, vc, vs, st, total;
};

WsLayout ws_layout(int B, int H, int N, int D) {
  const size_t BH = static_cast<size_t>(B) * H;
  const OperandSizes os = operand_sizes(N, D);
  WsLayout w;
  size_t off = 0;
  w.qc = off;
  off += align256(BH * os.q_codes);
  w.qs = off;
  off += align256(BH * os.q_scales);
  w.kc = off;
  off += align256(BH * os.q_codes);
  w.ks = off;
  off += align256(BH * os.q_scales);
  w.vc = off;
  off += align256(BH * os.vt_codes);
  w.vs = off;
  off += align256(BH * os.vt_scales);
  w.st = off;
  off += 256;
  w.total = off;
  return w;
}

bool tensor_ok(const sage_fp4_tensor& t) { return aligned(t.codes, 16) && aligned(t.scales, 16); }

bool qkv_ok(const sage_fp4_qkv* x) {
  return x && tensor_ok(x->q) && tensor_ok(x->k) && tensor_ok(x->vt) && aligned(x->status, 4);
}

// The kernels are compiled for sm_103a only.
int check_device() {
  static int cache[64];  // 0 unknown, 1 supported, 2 not
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

// 2-D byte tensor [rows][inner] (row pitch = inner), box [box_rows][box_inner].
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
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

CUtensorMapSwizzle swizzle_for_row(int row_bytes) {
  return row_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                         : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? SAGE_FP4_OK : SAGE_FP4_ECUDA; }

// bf16 elements addressable through a [B,H,N,D] tensor with strides s: its
// largest element offset + 1 (the strides were checked not to overflow)
long long tensor_extent(const Strides& s, int B, int H, int N, int D) {
  return static_cast<long long>(B - 1) * s.b + static_cast<long long>(H - 1) * s.h +
         static_cast<long long>(N - 1) * s.n + D;
}

// The sizes the debug build checks kernel indexes against (x[] and o as given).
Extents operand_extents(int32_t* status, int B, int H, int N, int D) {
  const OperandSizes os = operand_sizes(N, D);
  const long long BH = static_cast<long long>(B) * H;
  Extents e;
  e.status = status;
  e.x[0] = e.x[1] = e.x[2] = 0;
  e.o = 0;
  e.codes = BH * static_cast<long long>(os.q_codes);
  e.scales = BH * static_cast<long long>(os.q_scales);
  e.vt_codes = BH * static_cast<long long>(os.vt_codes);
  e.vt_scales = BH * static_cast<long long>(os.vt_scales);
  return e;
}

// Strides of one tensor: NULL means the contiguous [B,H,N,D] layout.  Each
// stride is >= 0 and a multiple of 8 elements (16-byte rows for the vector
// loads, bulk copies and stores), and the largest element offset fits in 62
// bits.
bool strides_of(const sage_fp4_strides* in, int B, int H, int N, int D, Strides* out) {
  if (!in) {
    *out = contiguous_bhnd(H, N, D);
    return true;
  }
  const int64_t st[3] = {in->b, in->h, in->n};
  const int64_t dims[3] = {B, H, N};
  int64_t last = D;
  for (int i = 0; i < 3; ++i) {
    if (st[i] < 0 || st[i] % 8 != 0) return false;
    int64_t span = 0;
    if (dims[i] > 0 && (__builtin_mul_overflow(st[i], dims[i] - 1, &span) ||
                        __builtin_add_overflow(last, span, &last)))
      return false;
  }
  if (last > (int64_t(1) << 62)) return false;
  *out = Strides{st[0], st[1], st[2]};
  return true;
}

bool scale_ok(float s) { return s > 0.0f && s <= 1.0e30f; }

bool format_ok(int f) {
  return f == SAGE_FP4_FORMAT_NVFP4 || f == SAGE_FP4_FORMAT_MXFP4 || f == SAGE_FP4_FORMAT_MXFP4_DIRECTP;
}

}  // namespace

extern "C" {

size_t sage_fp4_workspace_bytes(int B, int H, int N, int D) {
  if (!dims_ok(B, H, N, D)) return 0;
  return ws_layout(B, H, N, D).total;
}

int sage_fp4_qkv_from_workspace(void* workspace, size_t workspace_bytes, int B, int H, int N, int D,
                                sage_fp4_qkv* out) {
  if (!out || !dims_ok(B, H, N, D) || !aligned(workspace, 256)) return SAGE_FP4_EINVAL;
  const WsLayout w = ws_layout(B, H, N, D);
  if (workspace_bytes < w.total) return SAGE_FP4_EINVAL;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  out->q.codes = base + w.qc;
  out->q.scales = base + w.qs;
  out->k.codes = base + w.kc;
  out->k.scales = base + w.ks;
  out->vt.codes = base + w.vc;
  out->vt.scales = base + w.vs;
  out->status = reinterpret_cast<int32_t*>(base + w.st);
  return SAGE_FP4_OK;
}

namespace {

int quantize_impl(const void* q, const sage_fp4_strides* q_strides, const void* k,
                  const sage_fp4_strides* k_strides, const void* v, const sage_fp4_strides* v_strides,
                  const sage_fp4_qkv* out, int B, int H, int N, int D, int format, uint64_t wait_ns,
                  int withhold, void* stream) {
  if (!dims_ok(B, H, N, D) || !out || !format_ok(format)) return SAGE_FP4_EINVAL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return SAGE_FP4_EINVAL;
  if (!tensor_ok(out->q) || !tensor_ok(out->k) || !tensor_ok(out->vt) || !aligned(out->status, 4))
    return SAGE_FP4_EINVAL;
  Strides sq, sk, sv;
  if (!strides_of(q_strides, B, H, N, D, &sq) || !strides_of(k_strides, B, H, N, D, &sk) ||
      !strides_of(v_strides, B, H, N, D, &sv))
    return SAGE_FP4_EINVAL;
  if (is_empty(B, H, N)) return SAGE_FP4_OK;
  int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  const bool mx = format != SAGE_FP4_FORMAT_NVFP4;  // Direct-P operands are MXFP4
  Extents ext = operand_extents(out->status, B, H, N, D);
  ext.x[0] = tensor_extent(sq, B, H, N, D);
  ext.x[1] = tensor_extent(sk, B, H, N, D);
  ext.x[2] = tensor_extent(sv, B, H, N, D);
  cudaError_t e = launch_quant_rows(q, k, sq, sk, out->q.codes, out->q.scales, out->k.codes,
                                    out->k.scales, H, BH, N, D, mx, ext, st);
  if (e != cudaSuccess) return SAGE_FP4_ECUDA;
  return from_cuda(launch_quant_v(v, sv, out->vt.codes, out->vt.scales, H, BH, N, D, mx, out->status, wait_ns,
                                  withhold, ext, st));
}

}  // namespace

int sage_fp4_quantize_qkv_strided(const void* q, const sage_fp4_strides* q_strides, const void* k,
                                  const sage_fp4_strides* k_strides, const void* v,
                                  const sage_fp4_strides* v_strides, const sage_fp4_qkv* out, int B,
                                  int H, int N, int D, int format, void* stream) {
  return quantize_impl(q, q_strides, k, k_strides, v, v_strides, out, B, H, N, D, format, kAttnWaitNs, 0,
                       stream);
}

int sage_fp4_quantize_qkv_stall_test(const void* q, const void* k, const void* v, const sage_fp4_qkv* out,
                                     int B, int H, int N, int D, uint64_t wait_limit_ns, void* stream) {
  if (wait_limit_ns < 1000000ull || wait_limit_ns > kAttnWaitNs) return SAGE_FP4_EINVAL;
  return quantize_impl(q, nullptr, k, nullptr, v, nullptr, out, B, H, N, D, SAGE_FP4_FORMAT_NVFP4,
                       wait_limit_ns, 1, stream);
}

int sage_fp4_quantize_qkv(const void* q, const void* k, const void* v, const sage_fp4_qkv* out,
                          int B, int H, int N, int D, void* stream) {
  return sage_fp4_quantize_qkv_strided(q, nullptr, k, nullptr, v, nullptr, out, B, H, N, D,
                                       SAGE_FP4_FORMAT_NVFP4, stream);
}

namespace {

int attn_fwd_impl(const sage_fp4_qkv* qkv, void* o, const sage_fp4_strides* o_strides, int B, int H,
                  int N, int D, int causal, float scale, int format, int flags, uint64_t wait_ns,
                  void* stream) {
  if (!dims_ok(B, H, N, D) || !qkv_ok(qkv) || !aligned(o, 16) || !format_ok(format)) return SAGE_FP4_EINVAL;
  if (causal != 0 && causal != 1) return SAGE_FP4_EINVAL;
  Strides so;
  if (!strides_of(o_strides, B, H, N, D, &so) || !scale_ok(scale)) return SAGE_FP4_EINVAL;
  if (format == SAGE_FP4_FORMAT_MXFP4_DIRECTP) {
    const Strides dense = contiguous_bhnd(H, N, D);
    if (so.b != dense.b || so.h != dense.h || so.n != dense.n) return SAGE_FP4_EINVAL;
  }
  if (is_empty(B, H, N)) return SAGE_FP4_OK;
  int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  const int BH = B * H;
  const int Np = round_up_int(N, 128);
  CUtensorMap tq, tk, tv;
  const CUtensorMapSwizzle qk_swz = swizzle_for_row(D / 2);
  if (!make_map(&tq, qkv->q.codes, D / 2, static_cast<uint64_t>(BH) * Np, D / 2, 128, qk_swz) ||
      !make_map(&tk, qkv->k.codes, D / 2, static_cast<uint64_t>(BH) * Np, D / 2, 128, qk_swz) ||
      !make_map(&tv, qkv->vt.codes, Np / 2, static_cast<uint64_t>(BH) * D, 64, D,
                CU_TENSOR_MAP_SWIZZLE_64B))
    return SAGE_FP4_ECUDA;
  AttnParams p;
  p.sfq = qkv->q.scales;
  p.sfk = qkv->k.scales;
  p.sfv = qkv->vt.scales;
  p.o = o;
  p.os = so;
  p.status = qkv->status;
  p.H = H;
  p.BH = BH;
  p.N = N;
  p.Np = Np;
  p.causal = causal;
  p.n_qt = Np / 128;
  p.a = static_cast<float>(1.4426950408889634 * static_cast<double>(scale));
  p.mx = format == SAGE_FP4_FORMAT_MXFP4 ? 1 : format == SAGE_FP4_FORMAT_MXFP4_DIRECTP ? 2 : 0;
  p.flags = flags;
  p.wait_ns = wait_ns;
#if SAGE_FP4_DEBUG_BOUNDS
  p.ext = operand_extents(qkv->status, B, H, N, D);
  p.ext.o = tensor_extent(so, B, H, N, D);
#endif
  return from_cuda(launch_attn(tq, tk, tv, p, D, static_cast<cudaStream_t>(stream)));
}

// The softmax scale when the caller gives none: 1/sqrt(D).
float default_scale(int D) { return static_cast<float>(1.0 / sqrt(static_cast<double>(D > 0 ? D : 1))); }

}  // namespace

int sage_fp4_attn_fwd_ex(const sage_fp4_qkv* qkv, void* o, const sage_fp4_strides* o_strides, int B,
                         int H, int N, int D, int causal, float softmax_scale, int format,
                         void* stream) {
  return attn_fwd_impl(qkv, o, o_strides, B, H, N, D, causal, softmax_scale, format, 0, kAttnWaitNs,
                       stream);
}

int sage_fp4_attn_fwd(const sage_fp4_qkv* qkv, void* o, int B, int H, int N, int D, int causal,
                      void* stream) {
  return attn_fwd_impl(qkv, o, nullptr, B, H, N, D, causal, default_scale(D), SAGE_FP4_FORMAT_NVFP4, 0,
                       kAttnWaitNs, stream);
}

int sage_fp4_attn_fwd_stall_test(const sage_fp4_qkv* qkv, void* o, int B, int H, int N, int D,
                                 int causal, uint64_t wait_limit_ns, void* stream) {
  if (wait_limit_ns < 1000000ull || wait_limit_ns > kAttnWaitNs) return SAGE_FP4_EINVAL;
  return attn_fwd_impl(qkv, o, nullptr, B, H, N, D, causal, default_scale(D), SAGE_FP4_FORMAT_NVFP4,
                       kAttnWithholdK, wait_limit_ns, stream);
}

int sage_fp4_get_status(const sage_fp4_qkv* qkv, void* stream) {
  if (!qkv || !aligned(qkv->status, 4)) return SAGE_FP4_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SAGE_FP4_ECUDA;
  int32_t h = 0;
  if (cudaMemcpy(&h, qkv->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SAGE_FP4_ECUDA;
  if (h != 0 && cudaMemset(qkv->status, 0, sizeof(h)) != cudaSuccess) return SAGE_FP4_ECUDA;
  return h;
}

const char* sage_fp4_strerror(int status) {
  switch (status) {
    case SAGE_FP4_OK:
      return "ok";
    case SAGE_FP4_EINVAL:
      return "invalid argument (null or misaligned pointer, bad size, or D not 64/128)";
    case SAGE_FP4_ECUDA:
      return "CUDA runtime or driver error";
    case SAGE_FP4_ETIMEOUT:
      return "a kernel's bounded wait gave up; the output is not valid";
    case SAGE_FP4_EUNSUPPORTED:
      return "device is not sm_103 (kernels are built for sm_103a)";
    case SAGE_FP4_ETOOLARGE:
      return "problem needs more than the no-allocation entry's fixed 64 MiB scratch";
    case SAGE_FP4_EBOUNDS:
      return "debug build: a kernel computed an index outside its buffer (the access was skipped)";
    default:
      return "unknown status";
  }
}

int sage_fp4_cvt_probe(uint32_t first, uint32_t count, uint8_t* e2m1, uint8_t* e4m3,
                       void* stream) {
  if (!e2m1 && !e4m3) return SAGE_FP4_EINVAL;
  if (count == 0) return SAGE_FP4_OK;
  int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  return from_cuda(launch_cvt_probe(first, count, e2m1, e4m3, static_cast<cudaStream_t>(stream)));
}

namespace {

int mma_probe_impl(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* b_codes,
                   const uint8_t* b_scales, int n, int K, int flags, float* d, int32_t* status,
                   void* stream) {
  if (n != 64 && n != 128) return SAGE_FP4_EINVAL;
  if (flags & ~(SAGE_FP4_PROBE_A_BY_THREADS | SAGE_FP4_PROBE_MX | SAGE_FP4_PROBE_SF_ROWS128))
    return SAGE_FP4_EINVAL;
  if (K != 64 && K != 128 && K != 256) return SAGE_FP4_EINVAL;
  if (!aligned(a_codes, 16) || !aligned(a_scales, 16) || !aligned(b_codes, 16) ||
      !aligned(b_scales, 16) || !aligned(d, 4) || !aligned(status, 4))
    return SAGE_FP4_EINVAL;
  int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  CUtensorMap ta, tb;
  const CUtensorMapSwizzle swz = swizzle_for_row(K / 2);
  if (!make_map(&ta, a_codes, K / 2, 128, K / 2, 128, swz) ||
      !make_map(&tb, b_codes, K / 2, n, K / 2, n, swz))
    return SAGE_FP4_ECUDA;
  MmaProbeParams p;
  p.a_codes = a_codes;
  p.a_scales = a_scales;
  p.b_scales = b_scales;
  p.d = d;
  p.status = status;
  p.n = n;
  p.K = K;
  p.a_by_threads = (flags & SAGE_FP4_PROBE_A_BY_THREADS) ? 1 : 0;
  p.mx = (flags & SAGE_FP4_PROBE_MX) ? 1 : 0;
  p.sf_rows128 = (flags & SAGE_FP4_PROBE_SF_ROWS128) ? 1 : 0;
  return from_cuda(launch_mma_probe(ta, tb, p, static_cast<cudaStream_t>(stream)));
}

}  // namespace

int sage_fp4_mma_probe(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* b_codes,
                       const uint8_t* b_scales, int n, int K, int a_by_threads, float* d,
                       int32_t* status, void* stream) {
  return mma_probe_impl(a_codes, a_scales, b_codes, b_scales, n, K,
                        a_by_threads ? SAGE_FP4_PROBE_A_BY_THREADS : 0, d, status, stream);
}

int sage_fp4_mma_probe_ex(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* b_codes,
                          const uint8_t* b_scales, int n, int K, int flags, float* d, int32_t* status,
                          void* stream) {
  return mma_probe_impl(a_codes, a_scales, b_codes, b_scales, n, K, flags, d, status, stream);
}

int sage_fp4_mma_peak(int iters, int n, int32_t* status, void* stream) {
  if (iters < 1 || iters > 1000000 || (n != 128 && n != 256) || !aligned(status, 4)) return SAGE_FP4_EINVAL;
  int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  return from_cuda(launch_mma_peak(iters, n, status, static_cast<cudaStream_t>(stream)));
}

int sage_fp4_tmem_max_probe(const float* in, float* vals, float* maxes, void* stream) {
  if (!aligned(in, 16) || !aligned(vals, 16) || !aligned(maxes, 16)) return SAGE_FP4_EINVAL;
  int dev = check_device();
  if (dev != SAGE_FP4_OK) return dev;
  return from_cuda(launch_tmem_max_probe(in, vals, maxes, static_cast<cudaStream_t>(stream)));
}

int sage_fp4_mma_probe_mx(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* b_codes,
                          const uint8_t* b_scales, int n, int K, int a_by_threads, float* d,
                          int32_t* status, void* stream) {
  return mma_probe_impl(a_codes, a_scales, b_codes, b_scales, n, K,
                        SAGE_FP4_PROBE_MX | (a_by_threads ? SAGE_FP4_PROBE_A_BY_THREADS : 0), d, status,
                        stream);
}

}  // extern "C"

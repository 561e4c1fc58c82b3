// host_pipe.cu -- the whole path from host memory: bf16 Q, K, V in host
// memory -> bf16 O in host memory, with the host link kept busy.
//
// The GPU's link to host memory moves about 0.2 TB/s each way, so for the
// prefill shapes the copies take longer than the quantize and attention
// kernels together.  Done one after another (copy in, compute, copy out)
// the link idles while the kernels run and the SMs idle during the copies.
// sage_fp4_attention_host cuts the B*H heads into chunks and runs a
// three-stage pipeline over them, each stage on its own stream:
//
//   H2D stream      copy chunk i's q, k, v into staging slot i % 3
//   compute stream  quantize and attend chunk i (two calls of this library)
//   D2H stream      copy chunk i's O out of the slot
//
// so that chunk i+1 comes in and chunk i-1 goes out while chunk i computes.
// Attention and quantization treat every head on its own, so the result is
// bit-identical to one sage_fp4_quantize_qkv + sage_fp4_attn_fwd over the
// whole problem.
#include <cuda_runtime.h>
#include <limits.h>

#include <mutex>

#include "../../include/sage_fp4.h"
#include "layout.cuh"

using namespace sagefp4;

namespace {

constexpr int kSlots = 3;         // staging slots: in flight = copy-in, compute, copy-out
constexpr int kTargetChunks = 8;  // chunks per call when there are enough heads
constexpr int kMaxDevices = 64;

struct Plan {
  int BH = 0, c = 0, nchunks = 0;  // heads, heads per chunk, chunks
  size_t head_bytes = 0;           // bf16 bytes of one head of one tensor (N * D * 2)
  size_t stage = 0;                // bytes of one staged tensor in a slot (c heads, 256-aligned)
  size_t qws = 0;                  // quantized-operand workspace of one slot
  size_t slot = 0, total = 0;
};

bool plan_for(int B, int H, int N, int D, Plan* p) {
  if (B < 0 || H < 0 || N < 0 || (D != 64 && D != 128)) return false;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > INT_MAX) return false;
  p->BH = static_cast<int>(BH);
  p->head_bytes = static_cast<size_t>(N) * D * 2;
  if (BH == 0 || N == 0) return true;  // nothing to stage
  p->c = static_cast<int>((BH + kTargetChunks - 1) / kTargetChunks);
  p->nchunks = static_cast<int>((BH + p->c - 1) / p->c);
  p->qws = sage_fp4_workspace_bytes(1, p->c, N, D);
  if (p->qws == 0) return false;
  p->stage = align256(static_cast<size_t>(p->c) * p->head_bytes);
  p->slot = 4 * p->stage + align256(p->qws);
  p->total = kSlots * p->slot;
  return true;
}

// Streams and events of the pipeline, created once per device and kept until
// the process exits; one call at a time per device enqueues on them.
struct DevicePipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t in[kSlots] = {}, done[kSlots] = {}, out[kSlots] = {};
};

DevicePipe g_pipes[kMaxDevices];

cudaError_t init_pipe(DevicePipe& d) {
  if (d.ready) return cudaSuccess;
  cudaError_t e;
  if ((e = cudaStreamCreateWithFlags(&d.h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
  if ((e = cudaStreamCreateWithFlags(&d.comp, cudaStreamNonBlocking)) != cudaSuccess) return e;
  if ((e = cudaStreamCreateWithFlags(&d.d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
  if ((e = cudaEventCreateWithFlags(&d.start, cudaEventDisableTiming)) != cudaSuccess) return e;
  for (int s = 0; s < kSlots; ++s) {
    if ((e = cudaEventCreateWithFlags(&d.in[s], cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&d.done[s], cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&d.out[s], cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  d.ready = true;
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t sage_fp4_host_workspace_bytes(int B, int H, int N, int D) {
  Plan p;
  if (!plan_for(B, H, N, D, &p)) return 0;
  return p.total > 0 ? p.total : 256;
}

int sage_fp4_attention_host(const void* q, const void* k, const void* v, void* o, int B, int H,
                            int N, int D, int causal, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream) {
  Plan p;
  if (!plan_for(B, H, N, D, &p) || (causal != 0 && causal != 1)) return SAGE_FP4_EINVAL;
  if (!q || !k || !v || !o || !workspace || !status) return SAGE_FP4_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0 || reinterpret_cast<uintptr_t>(status) % 4 != 0)
    return SAGE_FP4_EINVAL;
  if (workspace_bytes < p.total) return SAGE_FP4_EINVAL;
  if (p.BH == 0 || N == 0) return SAGE_FP4_OK;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAGE_FP4_ECUDA;
  DevicePipe& d = g_pipes[dev];
  std::lock_guard<std::mutex> lock(d.mu);
  if (init_pipe(d) != cudaSuccess) return SAGE_FP4_ECUDA;

  // Carve the slots: staged q, k, v, o of c heads, then the quantized
  // operands, whose status pointer is replaced by the caller's status word.
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* sq[kSlots];
  uint8_t* sk[kSlots];
  uint8_t* sv[kSlots];
  uint8_t* so[kSlots];
  sage_fp4_qkv ops[kSlots];
  for (int s = 0; s < kSlots; ++s) {
    uint8_t* sb = base + s * p.slot;
    sq[s] = sb;
    sk[s] = sb + p.stage;
    sv[s] = sb + 2 * p.stage;
    so[s] = sb + 3 * p.stage;
    const int rc = sage_fp4_qkv_from_workspace(sb + 4 * p.stage, p.qws, 1, p.c, N, D, &ops[s]);
    if (rc != SAGE_FP4_OK) return rc;
    ops[s].status = status;
  }

  cudaStream_t user = static_cast<cudaStream_t>(stream);
  const auto* hq = static_cast<const uint8_t*>(q);
  const auto* hk = static_cast<const uint8_t*>(k);
  const auto* hv = static_cast<const uint8_t*>(v);
  auto* ho = static_cast<uint8_t*>(o);
  // fork: the pipeline's streams start after the caller's earlier work
  if (cudaEventRecord(d.start, user) != cudaSuccess || cudaStreamWaitEvent(d.h2d, d.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(d.comp, d.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(d.d2h, d.start, 0) != cudaSuccess)
    return SAGE_FP4_ECUDA;
  int last = 0;
  for (int i = 0; i < p.nchunks; ++i) {
    const int s = i % kSlots;
    const int h0 = i * p.c;
    const int ci = (p.BH - h0 < p.c) ? p.BH - h0 : p.c;
    const size_t off = static_cast<size_t>(h0) * p.head_bytes;
    const size_t bytes = static_cast<size_t>(ci) * p.head_bytes;
    // copy in once the slot's previous chunk has been quantized (its inputs read)
    if (i >= kSlots && cudaStreamWaitEvent(d.h2d, d.done[s], 0) != cudaSuccess) return SAGE_FP4_ECUDA;
    if (cudaMemcpyAsync(sq[s], hq + off, bytes, cudaMemcpyDefault, d.h2d) != cudaSuccess ||
        cudaMemcpyAsync(sk[s], hk + off, bytes, cudaMemcpyDefault, d.h2d) != cudaSuccess ||
        cudaMemcpyAsync(sv[s], hv + off, bytes, cudaMemcpyDefault, d.h2d) != cudaSuccess ||
        cudaEventRecord(d.in[s], d.h2d) != cudaSuccess)
      return SAGE_FP4_ECUDA;
    // compute once the inputs are in and the slot's previous O has gone out
    if (cudaStreamWaitEvent(d.comp, d.in[s], 0) != cudaSuccess) return SAGE_FP4_ECUDA;
    if (i >= kSlots && cudaStreamWaitEvent(d.comp, d.out[s], 0) != cudaSuccess) return SAGE_FP4_ECUDA;
    int rc = sage_fp4_quantize_qkv(sq[s], sk[s], sv[s], &ops[s], 1, ci, N, D, d.comp);
    if (rc != SAGE_FP4_OK) return rc;
    rc = sage_fp4_attn_fwd(&ops[s], so[s], 1, ci, N, D, causal, d.comp);
    if (rc != SAGE_FP4_OK) return rc;
    if (cudaEventRecord(d.done[s], d.comp) != cudaSuccess) return SAGE_FP4_ECUDA;
    // copy out
    if (cudaStreamWaitEvent(d.d2h, d.done[s], 0) != cudaSuccess ||
        cudaMemcpyAsync(ho + off, so[s], bytes, cudaMemcpyDefault, d.d2h) != cudaSuccess ||
        cudaEventRecord(d.out[s], d.d2h) != cudaSuccess)
      return SAGE_FP4_ECUDA;
    last = s;
  }
  // join: the caller's stream continues once the last O (and so every
  // earlier copy and kernel of this call) has completed
  return cudaStreamWaitEvent(user, d.out[last], 0) == cudaSuccess ? SAGE_FP4_OK : SAGE_FP4_ECUDA;
}

}  // extern "C"

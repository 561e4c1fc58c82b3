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
// The call is the two-call API run over that array: the array is carved by
// sage_fp4_qkv_from_workspace, the caller's status word replaces the
// workspace's, and sage_fp4_quantize_qkv and sage_fp4_attn_fwd do the rest,
// so every argument check and launch is theirs.
//
// That array is reserved on every GPU that loads this module and is held
// until the process exits.  Every call uses the same array: calls whose work
// overlaps on the GPU (different streams, or different host threads, without
// ordering between them) race on it and give undefined results.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/sage_fp4.h"

namespace {

constexpr size_t kScratchBytes = size_t(SAGE_FP4_NOALLOC_SCRATCH_BYTES);

// Quantized Q, K, V^T of the current call (and the workspace's unused status slot).
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

bool aligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The unique ID of the calling thread's current CUDA context (CUDA 12.0
// driver API, reached through the runtime's entry-point query).  IDs are never
// reused within a process, so a context created after cudaDeviceReset, or a
// second context on the same device, has an ID of its own.  False when no
// context is current or the query is unavailable.
bool current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch in the current context.  In host code g_scratch
// names a host-side stand-in, not device memory, so kernels must be given
// this address.  It is looked up with cudaGetSymbolAddress the first time a
// context calls (once per device in the usual one-context-per-device
// program) and kept, keyed by the context's unique ID, under a lock so that
// two threads' first calls do not race.
uint8_t* scratch_address() {
  struct Entry {
    unsigned long long ctx_id;
    uint8_t* addr;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int used = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  bool have_id = current_context_id(&id);
  if (have_id)
    for (int i = 0; i < used; ++i)
      if (cache[i].ctx_id == id) return cache[i].addr;
  // The lookup also makes the device's primary context current when the
  // runtime has not done so on this thread yet.
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return nullptr;
  if (!have_id) have_id = current_context_id(&id);
  if (have_id) {
    cache[next] = Entry{id, static_cast<uint8_t*>(p)};
    next = (next + 1) % 64;
    if (used < 64) ++used;
  }
  return static_cast<uint8_t*>(p);
}

}  // namespace

extern "C" int sage_fp4_attention_noalloc(const void* q, const void* k, const void* v, void* o,
                                          int32_t* status, int B, int H, int N, int D, int causal,
                                          void* stream) {
  // Sizes first: 0 means invalid sizes, anything above the array is too large.
  const size_t need = sage_fp4_workspace_bytes(B, H, N, D);
  if (need == 0 || (causal != 0 && causal != 1)) return SAGE_FP4_EINVAL;
  if (need > kScratchBytes) return SAGE_FP4_ETOOLARGE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(status, 4))
    return SAGE_FP4_EINVAL;
  if (static_cast<long long>(B) * H * N == 0) return SAGE_FP4_OK;
  uint8_t* base = scratch_address();
  if (!base) return SAGE_FP4_ECUDA;
  sage_fp4_qkv ops;
  int rc = sage_fp4_qkv_from_workspace(base, kScratchBytes, B, H, N, D, &ops);
  if (rc != SAGE_FP4_OK) return rc;
  ops.status = status;
  // Every byte of the quantized operands, padding included, is rewritten by
  // the quantize kernels, so nothing left by an earlier call is read.
  rc = sage_fp4_quantize_qkv(q, k, v, &ops, B, H, N, D, stream);
  if (rc != SAGE_FP4_OK) return rc;
  return sage_fp4_attn_fwd(&ops, o, B, H, N, D, causal, stream);
}

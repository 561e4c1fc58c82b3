// attn.cu -- fused NVFP4 attention forward for sm_103a (SageAttention3 method).
//
// A persistent CTA walks a fixed list of work items; an item is one tile of
// 128 query rows of one (batch, head), and it streams the item's KV tiles of
// 128 keys.  The KV tiles of all the CTA's items form one stream g = 0, 1, ...
// that every role walks in the same order, so the next item's first tiles
// overlap the current item's last ones.  Per KV tile:
//   S   = (Q^ sQ)(K^ sK)^T     block-scaled FP4 tensor-core MMA into tensor memory
//   online softmax over S fused with two-level P quantization: level 1 maps
//       the tile's row segment onto [0, 448*6] (its maximum becomes 2688),
//       level 2 quantizes 1x16 groups along keys to NVFP4; the 16-element
//       maxima double as the row maximum (senqingzn.com article on
//       SageAttention3, "Solving two obstacles and one difficulty", solution
//       2; "FP4 attention inference acceleration and hardware
//       implementation/optimisation", fusion paragraph)
//   PV  = (P^ sP)(V^ sV)        block-scaled FP4 MMA with FP32 accumulation
//   O   = O * exp(m_old - m_new) + exp(t - m_new)/2688 * PV   (FP32)
// Roles (warp specialisation, mbarrier pipelines, all waits bounded):
//   warp 0       bulk-copy producer of Q and K tiles and their scales
//   warp 1       tcgen05 issuer of S = QK^T (one thread)
//   warp 2       tensor-memory allocator, then producer of V^T tiles
//   warp 3       tcgen05 issuer of PV (one thread)
//   warps 4-7    softmax + P quantization of the even tiles g, one thread per row
//   warps 8-11   the same for the odd tiles: with level 1 normalised per
//                tile, tiles are independent until O is combined
//   warps 12-15  correction: rescale-and-accumulate O in registers, epilogue
// Tensor memory (512 columns x 128 lanes): each softmax warpgroup owns one
// 128-column S buffer, which it hands back to the S issuer as soon as it has
// loaded its rows, so the next S of that warpgroup overlaps the rest of its
// softmax.  PV goes through separate buffers that the correction empties (one
// of 128 columns at D = 128, three of 64 at D = 64), so the correction is off
// the S buffers' loop.  The last 64 columns hold double-buffered scale
// factors of Q, K, V and P.  Every MMA group ends in exactly one
// tcgen05.commit (each costs ~40 cycles of issue and ~250 cycles until the
// barrier is seen on GB300).
// Registers are rebalanced with setmaxnreg (budgets per head dimension below).
// Instantiations: D (64, 128) x O layout (dense [B,H,N,D], or through
// strides) x format (NVFP4, the method's; MXFP4, 1x32 groups with E8M0
// scales, the alternative the pages set aside -- its level 1 targets 6).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "../../include/sage_fp4.h"
#include "kernels.h"
#include "layout.cuh"
#include "ptx.cuh"

namespace sagefp4 {

namespace {

constexpr int kStages = 6;   // K and V^T shared-memory ring depth
constexpr int kPSlots = 3;   // P tiles (and their scales) in shared memory
constexpr int kEvRing = 6;   // P and row-stat events: slot g % 6
constexpr int kPvBufsMax = 3;  // PV buffers (D = 64: three of 64 columns; D = 128: one of 128)
constexpr int kPvRing = 12;  // PV completion events
constexpr int kThreads = 512;
// Register budgets (setmaxnreg) of the control warps, each softmax thread and
// each correction thread.  The correction holds its O row (D registers) plus
// 64 columns of PV, so that it waits once per 64 columns of a PV buffer; at
// D = 128 that costs the softmax 16 registers (measured net gain 4-6%).
template <int D>
struct Regs;
template <>
struct Regs<128> {
  static constexpr uint32_t kCtl = 48, kSoftmax = 128, kCorr = 208;
};
template <>
struct Regs<64> {
  static constexpr uint32_t kCtl = 48, kSoftmax = 144, kCorr = 176;
};
static_assert(Regs<128>::kCtl * 128 + Regs<128>::kSoftmax * 256 + Regs<128>::kCorr * 128 == 65536, "split");
static_assert(Regs<64>::kCtl * 128 + Regs<64>::kSoftmax * 256 + Regs<64>::kCorr * 128 == 65536, "split");
constexpr unsigned kFull = 0xFFFFFFFFu;

// tensor-memory columns
constexpr uint32_t kColS = 0;      // 2 S buffers x 128 (buffer = softmax warpgroup)
constexpr uint32_t kColPV = 256;   // PV buffers: 1 x 128 (D = 128) or 3 x 64 (D = 64)
constexpr uint32_t kColSFQ = 448;  // 2 item slots x 8
constexpr uint32_t kColSFK = 464;  // 2 slots x 8
constexpr uint32_t kColSFV = 480;  // 2 slots x 8
constexpr uint32_t kColSFP = 496;  // 2 slots x 8
constexpr uint32_t kTmemCols = 512;

// barrier indices.  A barrier of a ring of R serves events n = i, i+R, ...;
// the waiter for event n waits for completion number n / R (parity (n/R)&1).
// PV is event e = g (one MMA group per tile).
enum {
  B_QFULL = 0,                     // Q tile of local item i landed          [2]
  B_QEMPTY = B_QFULL + 2,          // every S of local item i completed      [2]
  B_KFULL = B_QEMPTY + 2,          // K_g landed                             [kStages]
  B_VFULL = B_KFULL + kStages,     // V_g landed                             [kStages]
  B_SDONE = B_VFULL + kStages,     // S_g in tensor memory, K slot free      [kStages]
  B_SFREE = B_SDONE + kStages,     // S buffer w read by its softmax         [2]
  B_PFULL = B_SFREE + 2,           // P_g, its scales and row stats written  [kEvRing]
  B_PVDONE = B_PFULL + kEvRing,    // PV_e in tensor memory                  [kPvRing]
  B_PVFREE = B_PVDONE + kPvRing,   // PV buffer read by the correction       [kPvBufsMax]
  B_DRAIN = B_PVFREE + kPvBufsMax,    // abandoning work: MMAs of one issuer   [2]
  kNumBars = B_DRAIN + 2
};

template <int D>
struct Smem {
  static constexpr int KBD = D / 64;           // 64-element K blocks along D
  static constexpr int QBYTES = 128 * D / 2;   // Q or K code tile (128 rows)
  static constexpr int SFQK = KBD * 512;       // scales of one Q or K tile
  static constexpr int VBYTES = D * 64;        // V^T code tile: D rows x 128 keys
  static constexpr int SFVB = 1024;            // V^T scales of one tile (2 K-blocks)
  static constexpr int PBYTES = 128 * 64;      // P code tile: 128 rows x 128 keys
  // P scales of one tile.  At D = 64 the softmax writes them as the source of
  // one 128-lane copy (row r's word of each 64-key step at lane r, column
  // base + r / 32, the layout the MMA reads for its A operand): 4 KB, one copy
  // instead of two (measured +2% at D = 64, -0.5% at D = 128).  At D = 128
  // they stay in the 512-byte-per-step block layout, copied replicated.
  static constexpr int SFPB = (D == 64) ? 4096 : 1024;
  // swizzled tiles first (every one a multiple of 1 KB from a 1 KB-aligned base)
  static constexpr int oQ = 0;
  static constexpr int oK = oQ + 2 * QBYTES;
  static constexpr int oV = oK + kStages * QBYTES;
  static constexpr int oP = oV + kStages * VBYTES;
  static constexpr int oSFQ = oP + kPSlots * PBYTES;
  static constexpr int oSFK = oSFQ + 2 * SFQK;
  static constexpr int oSFV = oSFK + kStages * SFQK;
  static constexpr int oSFP = oSFV + kStages * SFVB;
  static constexpr int oStat = oSFP + kPSlots * SFPB;
  static constexpr int oLut = oStat + kEvRing * 128 * 8;  // float2 per E4M3 byte
  static constexpr int oBar = oLut + 256 * 8;
  static constexpr int oMisc = oBar + kNumBars * 8;
  static constexpr int kBytes = oMisc + 16;
  // 1 KB slack to align the base; at least 120 KB so that one CTA owns an SM
  // (the CTA allocates all 512 tensor-memory columns)
  static constexpr int kAlloc = (kBytes + 1024 > 120 * 1024) ? kBytes + 1024 : 120 * 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

struct Ctl {
  volatile int* abort;
  int32_t* status;
  uint64_t limit;  // ns after which a bounded wait gives up
};

__device__ __forceinline__ void give_up(const Ctl& c) {
  *c.abort = 1;
  atomicCAS(c.status, 0, SAGE_FP4_ETIMEOUT);
}

// Bounded wait by a single thread.  False: the CTA is abandoning its work.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, Ctl c) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if (globaltimer_ns() - t0 > c.limit) {
      give_up(c);
      return false;
    }
  }
}

// Bounded wait by a whole warp; every lane gets the same answer.
__device__ __forceinline__ bool waitw(uint32_t bar, uint32_t parity, Ctl c) {
  if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
    int stop = 0;
    if ((threadIdx.x & 31) == 0) {
      if (*c.abort) {
        stop = 1;
      } else if (globaltimer_ns() - t0 > c.limit) {
        give_up(c);
        stop = 1;
      }
    }
    if (__shfl_sync(kFull, stop, 0)) return false;
  }
}

// Wait used only while abandoning work: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const Ctl& c) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < c.limit) {
  }
}

// All threads of the CTA, each role from its own code path (named barrier 1).
__device__ __forceinline__ void cta_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

constexpr float kLog2of2688 = 11.392317422778761f;  // log2(448 * 6)
constexpr float kLog2of448 = 8.807354922057604f;    // log2(448)

__device__ __forceinline__ float2 lds_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}
constexpr float kLog2of6 = 2.5849625007211563f;     // log2(6): the MXFP4 level-1 target

__device__ __forceinline__ float max16(const uint32_t* s) {
  auto f = [&](int i) { return __uint_as_float(s[i]); };
  const float m0 = max3f(f(0), f(1), f(2)), m1 = max3f(f(3), f(4), f(5));
  const float m2 = max3f(f(6), f(7), f(8)), m3 = max3f(f(9), f(10), f(11));
  const float m4 = max3f(f(12), f(13), f(14));
  return max3f(max3f(m0, m1, m2), max3f(m3, m4, f(15)), m0);
}

// Direct-P normaliser: the eight E2M1 codes of a word decoded (two per
// instruction) and summed as an f16 pair, lanes = even / odd codes.  Exact:
// the values are multiples of 1/2 and at most 6, so a lane's sum is a
// multiple of 1/2 no larger than 24.
__device__ __forceinline__ uint32_t e2m1x8_sum_h2(uint32_t w) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
      "add.rn.f16x2 h0, h0, h1;\n\t"
      "add.rn.f16x2 h2, h2, h3;\n\t"
      "add.rn.f16x2 %0, h0, h2;\n\t}"
      : "=r"(r)
      : "r"(w));
  return r;
}

// The sum of the two f16 halves of a pair, as FP32 (exact for the sums above).
__device__ __forceinline__ float h2_total(uint32_t a, uint32_t b) {
  uint32_t s;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(s) : "r"(a), "r"(b));
  float lo, hi;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(s));
  return lo + hi;
}

// A work item: 128 query rows (tile qt) of head bh and its nkv KV tiles.
// Causal lists start with the longest rows so that the static round-robin
// over CTAs stays balanced.
struct Item {
  int bh, qt, nkv;
};

__device__ __forceinline__ Item item_at(const AttnParams& p, int it) {
  Item r;
  if (p.causal) {
    r.qt = p.n_qt - 1 - it / p.BH;
    r.bh = it % p.BH;
    r.nkv = r.qt + 1;
  } else {
    r.bh = it / p.n_qt;
    r.qt = it % p.n_qt;
    r.nkv = p.Np / kTileKV;
  }
  return r;
}

// kMx: operands and P in MXFP4 (groups of 32, E8M0 scales) instead of NVFP4.
// kDirectP (with kMx): the row sum l is summed from the rounded P, the
// decoded codes times their scales, the same values PV uses (Direct-P, the
// rit.work summary of "Hardware-Aware FP4 FlashAttention-4", "Что
// сделали"), instead of from the unquantized exponentials.
template <int D, bool kDenseO, bool kMx, bool kDirectP = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using L = Smem<D>;
  constexpr int NH = 1;                    // PV groups per tile
  constexpr int kPvBufs = (D == 128) ? 1 : 3;  // PV buffers of D columns
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sb + L::oBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::oMisc + 4);
  const Ctl ctl{abort_flag, p.status, p.wait_ns};
  const int n_items = p.BH * p.n_qt;
  const int item0 = static_cast<int>(blockIdx.x), istep = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QFULL + s), 1);
      mbar_init(bar(B_QEMPTY + s), 1);
      mbar_init(bar(B_DRAIN + s), 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_SDONE + s), 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(bar(B_SFREE + s), 128);
    for (int s = 0; s < kEvRing; ++s) mbar_init(bar(B_PFULL + s), 128);
    for (int s = 0; s < kPvRing; ++s) mbar_init(bar(B_PVDONE + s), 1);
    for (int s = 0; s < kPvBufsMax; ++s) mbar_init(bar(B_PVFREE + s), 128);
    // a launch sharing this status word already gave up: do no work
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(p.status) != 0) ? 1 : 0;
    mbar_fence_init();
  }
  // Per E4M3 scale byte b of a P group: (log2(2688) - log2(value(b)), value(b) / 2688),
  // and (0, 1) for b = 0, whose group keeps the row's own bias.
  for (int b = threadIdx.x; b < 256; b += kThreads) {
    float x = 0.0f, y = 1.0f;
    if (b > 0 && b < 0x7F) {
      const float v = e4m3_to_f32(static_cast<uint32_t>(b));
      x = kLog2of2688 - log2f(v);
      y = v * (1.0f / 2688.0f);
    }
    reinterpret_cast<float2*>(sm + L::oLut)[b] = make_float2(x, y);
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;

  const int wg = warp / 4;
  if (wg == 0) {
    regs_dec<Regs<D>::kCtl>();
    if (!skip && warp == 0 && lane == 0) {
      // ---------------------------------------------------- Q and K producer
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      int nq = 0, nk = 0;  // copies issued
      bool ok = true;
      auto load_q = [&](int i, const Item& it) -> bool {
        const int s = i & 1;
        if (i >= 2 && !wait1(bar(B_QEMPTY + s), ((i >> 1) - 1) & 1, ctl)) return false;
        mbar_arrive_expect_tx(bar(B_QFULL + s), L::QBYTES + L::SFQK);
        tma_load_2d(sb + L::oQ + s * L::QBYTES, &tm_q, 0, it.bh * p.Np + it.qt * kTileQ, bar(B_QFULL + s));
#if SAGE_FP4_DEBUG_BOUNDS
        // debug build: a copy that would leave its buffer is skipped; the wait
        // for it then runs out after the bounds failure was recorded
        const long long qso = static_cast<long long>(it.bh) * p.Np * (D / 16) + static_cast<long long>(it.qt) * L::SFQK;
        if (in_bounds(p.ext, qso, L::SFQK, p.ext.scales))
          bulk_load(sb + L::oSFQ + s * L::SFQK, p.sfq + qso, L::SFQK, bar(B_QFULL + s));
#else
        bulk_load(sb + L::oSFQ + s * L::SFQK,
                  p.sfq + static_cast<size_t>(it.bh) * p.Np * (D / 16) + static_cast<size_t>(it.qt) * L::SFQK,
                  L::SFQK, bar(B_QFULL + s));
#endif
        nq = i + 1;
        return true;
      };
      int g = 0, i = 0;
      if (item0 < n_items) ok = load_q(0, item_at(p, item0));
      for (int it = item0; ok && it < n_items; it += istep, ++i) {
        const Item I = item_at(p, it);
        const uint8_t* sfk = p.sfk + static_cast<size_t>(I.bh) * p.Np * (D / 16);
        for (int k = 0; k < I.nkv; ++k, ++g) {
          const int s = g % kStages;
          if ((p.flags & kAttnWithholdK) && g >= 1) {
            ok = false;  // failure-detection test: the next K tile never comes
            break;
          }
          if (g >= kStages && !(ok = wait1(bar(B_SDONE + s), ((g / kStages) - 1) & 1, ctl))) break;
          mbar_arrive_expect_tx(bar(B_KFULL + s), L::QBYTES + L::SFQK);
          tma_load_2d(sb + L::oK + s * L::QBYTES, &tm_k, 0, I.bh * p.Np + k * kTileKV, bar(B_KFULL + s));
#if SAGE_FP4_DEBUG_BOUNDS
          if (in_bounds(p.ext, (sfk - p.sfk) + static_cast<long long>(k) * L::SFQK, L::SFQK, p.ext.scales))
#endif
            bulk_load(sb + L::oSFK + s * L::SFQK, sfk + static_cast<size_t>(k) * L::SFQK, L::SFQK,
                      bar(B_KFULL + s));
          nk = g + 1;
          // the next item's Q goes out once a few of this item's tiles are
          // queued (by then the item before this one has finished its S)
          if (k == min(kStages - 2, I.nkv - 1) && it + istep < n_items &&
              !(ok = load_q(i + 1, item_at(p, it + istep))))
            break;
        }
      }
      // every copy this thread started has landed before the CTA exits (at
      // once after a normal run; after a role gave up, possibly not yet)
      (void)ok;
      for (int j = (nq > 2 ? nq - 2 : 0); j < nq; ++j) drain_wait(bar(B_QFULL + (j & 1)), (j >> 1) & 1, ctl);
      for (int j = (nk > kStages ? nk - kStages : 0); j < nk; ++j)
        drain_wait(bar(B_KFULL + j % kStages), (j / kStages) & 1, ctl);
    } else if (!skip && warp == 2 && lane == 0) {
      // -------------------------------------------------------- V producer
      prefetch_tensormap(&tm_v);
      int nv = 0;
      bool ok = true;
      int g = 0;
      for (int it = item0; ok && it < n_items; it += istep) {
        const Item I = item_at(p, it);
        const uint8_t* sfv = p.sfv + static_cast<size_t>(I.bh) * 8 * p.Np;
        for (int k = 0; k < I.nkv; ++k, ++g) {
          const int s = g % kStages;
          if (g >= kStages) {
            const int e = (g - kStages) * NH + NH - 1;  // PV of tile g-6
            if (!(ok = wait1(bar(B_PVDONE + e % kPvRing), (e / kPvRing) & 1, ctl))) break;
          }
          mbar_arrive_expect_tx(bar(B_VFULL + s), L::VBYTES + L::SFVB);
          tma_load_2d(sb + L::oV + s * L::VBYTES, &tm_v, k * (kTileKV / 2), I.bh * D, bar(B_VFULL + s));
#if SAGE_FP4_DEBUG_BOUNDS
          if (in_bounds(p.ext, (sfv - p.sfv) + static_cast<long long>(k) * L::SFVB, L::SFVB, p.ext.vt_scales))
#endif
            bulk_load(sb + L::oSFV + s * L::SFVB, sfv + static_cast<size_t>(k) * L::SFVB, L::SFVB,
                      bar(B_VFULL + s));
          nv = g + 1;
        }
      }
      (void)ok;
      for (int j = (nv > kStages ? nv - kStages : 0); j < nv; ++j)
        drain_wait(bar(B_VFULL + j % kStages), (j / kStages) & 1, ctl);
    } else if (!skip && warp == 1 && lane == 0) {
      // ------------------------------------------------------- S issuer
      constexpr uint32_t idS = kMx ? idesc_mxf4(128, 128) : idesc_nvfp4(128, 128);
      constexpr uint32_t qk_swz = (D == 128) ? kSwizzle64B : kSwizzle32B;
      constexpr uint32_t qk_sbo = 8 * (D / 2);
      bool ok = true;
      int g = 0, i = 0;
      for (int it = item0; ok && it < n_items; it += istep, ++i) {
        const Item I = item_at(p, it);
        const int qs = i & 1;
        if (!(ok = wait1(bar(B_QFULL + qs), (i >> 1) & 1, ctl))) break;
        bool first = true;
        for (int k = 0; k < I.nkv; ++k, ++g) {
          const int s = g % kStages, w = g & 1, sl = g & 1;
          if (!(ok = wait1(bar(B_KFULL + s), (g / kStages) & 1, ctl))) break;
          // the scale factors go in while the softmax still reads the S buffer
          tc_fence_after();
          if (first) {
#pragma unroll
            for (int kb = 0; kb < L::KBD; ++kb)
              tc_cp_32x128b_warpx4(tmem + kColSFQ + 8 * qs + 4 * kb,
                                   smem_desc(sb + L::oSFQ + qs * L::SFQK + 512 * kb, 0, 128, kSwizzleNone));
            first = false;
          }
#pragma unroll
          for (int kb = 0; kb < L::KBD; ++kb)
            tc_cp_32x128b_warpx4(tmem + kColSFK + 8 * sl + 4 * kb,
                                 smem_desc(sb + L::oSFK + s * L::SFQK + 512 * kb, 0, 128, kSwizzleNone));
          // S buffer w is free once its softmax warpgroup has loaded S_{g-2}
          if (g >= 2 && !(ok = wait1(bar(B_SFREE + w), ((g >> 1) - 1) & 1, ctl))) break;
          tc_fence_after();
#pragma unroll
          for (int kb = 0; kb < L::KBD; ++kb) {
            const uint64_t ad = smem_desc(sb + L::oQ + qs * L::QBYTES + 32 * kb, 16, qk_sbo, qk_swz);
            const uint64_t bd = smem_desc(sb + L::oK + s * L::QBYTES + 32 * kb, 16, qk_sbo, qk_swz);
            if constexpr (kMx)
              mma_mxf4(tmem + kColS + w * 128, ad, bd, idS, tmem + kColSFQ + 8 * qs + 4 * kb,
                       tmem + kColSFK + 8 * sl + 4 * kb, kb > 0);
            else
              mma_nvfp4(tmem + kColS + w * 128, ad, bd, idS, tmem + kColSFQ + 8 * qs + 4 * kb,
                        tmem + kColSFK + 8 * sl + 4 * kb, kb > 0);
          }
          tc_commit(bar(B_SDONE + s));
        }
        if (ok) tc_commit(bar(B_QEMPTY + qs));
      }
      // the last item's release must land before the CTA can exit
      if (ok && i > 0) ok = wait1(bar(B_QEMPTY + ((i - 1) & 1)), ((i - 1) >> 1) & 1, ctl);
      // the tensor-core work this thread issued has completed before tensor
      // memory is freed (at once after a normal run)
      tc_commit(bar(B_DRAIN));
      drain_wait(bar(B_DRAIN), 0, ctl);
    } else if (!skip && warp == 3 && lane == 0) {
      // ------------------------------------------------------ PV issuer
      // PV_g (N = D) into the next PV buffer.  The loop over h is written for
      // groups of 64 output columns (V^T rows 64h.., whose scale factors sit
      // 2h columns further along: each column holds 32 rows); one group of
      // N = D is used, measured faster than two of 64 at D = 128.
      constexpr uint32_t idPV = kMx ? idesc_mxf4(128, D) : idesc_nvfp4(128, D);
      bool ok = true;
      int g = 0;
      for (int it = item0; ok && it < n_items; it += istep) {
        const int nkv = item_at(p, it).nkv;
        for (int k = 0; k < nkv; ++k, ++g) {
          const int s = g % kStages, ps = g % kPSlots, sl = g & 1;
          if (!(ok = wait1(bar(B_PFULL + g % kEvRing), (g / kEvRing) & 1, ctl))) break;
          if (!(ok = wait1(bar(B_VFULL + s), (g / kStages) & 1, ctl))) break;
          // the scale factors go in while the correction still reads the PV buffer
          tc_fence_after();
          if constexpr (D == 64) {
            // both steps' P scales in one copy (second 16 bytes of a row 2 KB on)
            tc_cp_128x256b(tmem + kColSFP + 8 * sl,
                           smem_desc(sb + L::oSFP + ps * L::SFPB, 2048, 128, kSwizzleNone));
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
              tc_cp_32x128b_warpx4(tmem + kColSFV + 8 * sl + 4 * kb,
                                   smem_desc(sb + L::oSFV + s * L::SFVB + 512 * kb, 0, 128, kSwizzleNone));
          } else {
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
              tc_cp_32x128b_warpx4(tmem + kColSFP + 8 * sl + 4 * kb,
                                   smem_desc(sb + L::oSFP + ps * L::SFPB + 512 * kb, 0, 128, kSwizzleNone));
              tc_cp_32x128b_warpx4(tmem + kColSFV + 8 * sl + 4 * kb,
                                   smem_desc(sb + L::oSFV + s * L::SFVB + 512 * kb, 0, 128, kSwizzleNone));
            }
          }
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int e = g * NH + h, pb = e % kPvBufs;
            if (e >= kPvBufs && !(ok = wait1(bar(B_PVFREE + pb), ((e / kPvBufs) - 1) & 1, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
              const uint64_t ad = smem_desc(sb + L::oP + ps * L::PBYTES + 32 * kb, 16, 512, kSwizzle64B);
              const uint64_t bd =
                  smem_desc(sb + L::oV + s * L::VBYTES + h * 64 * 64 + 32 * kb, 16, 512, kSwizzle64B);
              if constexpr (kMx)
                mma_mxf4(tmem + kColPV + pb * D, ad, bd, idPV, tmem + kColSFP + 8 * sl + 4 * kb,
                         tmem + kColSFV + 8 * sl + 4 * kb + 2 * h, kb > 0);
              else
                mma_nvfp4(tmem + kColPV + pb * D, ad, bd, idPV, tmem + kColSFP + 8 * sl + 4 * kb,
                          tmem + kColSFV + 8 * sl + 4 * kb + 2 * h, kb > 0);
            }
            tc_commit(bar(B_PVDONE + e % kPvRing));
          }
          if (!ok) break;
        }
      }
      tc_commit(bar(B_DRAIN + 1));
      drain_wait(bar(B_DRAIN + 1), 0, ctl);
    }
    // every role ends at the same CTA-wide barrier; then tensor memory is freed
    tc_fence_before();
    cta_bar_sync();
    if (warp == 2) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
  } else if (wg == 1 || wg == 2) {
    // -------------------------------------------------------- softmax + P quantization
    regs_inc<Regs<D>::kSoftmax>();
    if (!skip) {
      const int par = wg - 1;                // this warpgroup takes the tiles g with g % 2 == par
      const int r = threadIdx.x - 128 * wg;  // query row of this thread = TMEM lane
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const float a = p.a;
      const uint64_t a2 = pack2(a, a);
      const int sw = (r >> 1) & 3;  // 64-byte swizzle: 16-byte chunk c lives at c ^ ((r/2) % 4)
      const uint32_t lut = sb + L::oLut;
      bool ok = true;
      int g0 = 0;  // stream index of the current item's first tile
      for (int it = item0; ok && it < n_items; it += istep) {
        const Item I = item_at(p, it);
        const int gi = I.qt * kTileQ + r;
        const int vis_end = p.causal ? min(p.N, gi + 1) : p.N;  // keys j < vis_end are visible
        for (int k = (par - g0) & 1; k < I.nkv; k += 2) {
          const int g = g0 + k;
          const int lim = vis_end - k * kTileKV;  // keys of this tile at or past lim are invisible
          // One 128x128 tile.  The copy that masks keys (the causal diagonal,
          // the ragged end of N) is separate, so that every other tile runs a
          // shorter body (measured +6-12%: the warps stall on instruction fetch).
          auto tile = [&](auto masked_tag) -> bool {
            constexpr bool kMasked = decltype(masked_tag)::value;
            const int ps = g % kPSlots;
            if (!waitw(bar(B_SDONE + g % kStages), (g / kStages) & 1, ctl)) return false;
            tc_fence_after();
            const uint32_t tb = tmem + kColS + par * 128 + lane_base;
            // pass 1: the 16-element group maxima, whose maximum is the tile
            // maximum; the second 64 keys stay in registers for pass 2.  Where
            // no key is masked, each group's maximum comes with its load from
            // tensor memory (the reducing form of tcgen05.ld), with no
            // comparisons in the thread.
            float gm[8];
            uint32_t s64[64];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if constexpr (kMasked) {
                tmem_ld32(tb + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&s64[0]));
                tmem_ld32(tb + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&s64[32]));
                tmem_wait_ld();
                if (lim < kTileKV) {
#pragma unroll
                  for (int j = 0; j < 64; ++j)
                    if (64 * h + j >= lim) s64[j] = __float_as_uint(-INFINITY);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) gm[4 * h + q] = max16(&s64[16 * q]);
              } else {
                // groups whose maximum comes with the load: all eight at D = 64;
                // at D = 128 the first three (with four or more the kernel
                // spills registers and runs 7-12% slower; with three it gains
                // 2.7%, measured), the others by comparisons in the thread
                constexpr int kRedFirst = (D == 64) ? 4 : 3, kRedSecond = (D == 64) ? 4 : 0;
                const int nred = (h == 0) ? kRedFirst : kRedSecond;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  if (q < nred)
                    tmem_ld16_max(tb + 64 * h + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&s64[16 * q]),
                                  gm[4 * h + q]);
                  else
                    tmem_ld16(tb + 64 * h + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&s64[16 * q]));
                }
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  if (q >= nred) gm[4 * h + q] = max16(&s64[16 * q]);
              }
            }
            const float t = max3f(max3f(gm[0], gm[1], gm[2]), max3f(gm[3], gm[4], gm[5]),
                                  fmaxf(gm[6], gm[7]));
            const float nb = -t * a;
            // level 2 scale of each group from its maximum: E4M3(2688 e^(c(g - t)) / 6);
            // the code of element j is E2M1(2688 e^(c(S_j - t)) / scale), computed
            // as exp2(a S_j + bias_g); a group whose scale is 0 keeps bias nb so
            // that its (vanishing) probabilities still enter the row sum exactly
            float bias[8], lsc[8];
            uint32_t s2[4];  // scale bytes of 16-key groups (2i, 2i+1), two per 16 bits
            if constexpr (kMx) {
              // MXFP4: level 1 maps the row maximum to 6; each 32-key group's
              // E8M0 scale comes from its largest P2 = 6 exp2(a (S - t)), and
              // both 16-key halves take its bias (scale words: [e(2k), e(2k+1), 0, 0])
              uint32_t e8[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float p2 = 6.0f * ex2_approx(fmaf(fmaxf(gm[2 * j], gm[2 * j + 1]), a, nb));
                e8[j] = e8m0_of(p2);
                const float sh = static_cast<float>(static_cast<int>(e8[j]) - 127);
                bias[2 * j] = bias[2 * j + 1] = nb + (kLog2of6 - sh);
                lsc[2 * j] = lsc[2 * j + 1] = __uint_as_float(e8[j] << 23) * (1.0f / 6.0f);
              }
              s2[0] = e8[0] | (e8[1] << 8);
              s2[1] = 0u;
              s2[2] = e8[2] | (e8[3] << 8);
              s2[3] = 0u;
            } else {
              const float nbs = nb + kLog2of448;  // 448 e^(c(g - t)) as one exponential
#pragma unroll
              for (int q = 0; q < 8; q += 2) {
                const float e0 = ex2_approx(fmaf(gm[q], a, nbs));
                const float e1 = ex2_approx(fmaf(gm[q + 1], a, nbs));
                s2[q / 2] = cvt_e4m3x2(e0, e1);
                const float2 t0 = lds_f32x2(lut + 8 * (s2[q / 2] & 0xFFu)), t1 = lds_f32x2(lut + 8 * (s2[q / 2] >> 8));
                bias[q] = nb + t0.x;
                lsc[q] = t0.y;
                bias[q + 1] = nb + t1.x;
                lsc[q + 1] = t1.y;
              }
            }
            // P slot ps is free once PV_{g-3} has completed
            if (g >= kPSlots) {
              const int e = (g - kPSlots) * NH + NH - 1;
              if (!waitw(bar(B_PVDONE + e % kPvRing), (e / kPvRing) & 1, ctl)) return false;
            }
            uint8_t* prow = sm + L::oP + ps * L::PBYTES + r * 64;
            uint64_t acc[2] = {0ull, 0ull};  // row sum, two FP32x2 chains
            float rsum = 0.0f;               // Direct-P: row sum of the rounded P
            // pass 2: exponentials, row sum and codes, 64 keys per tensor-memory
            // wait.  Where registers allow (D = 64), keys 64-127 are still in
            // registers from pass 1 and go first; otherwise both halves are read
            // again in order.
            constexpr bool kKeep = (D == 64);
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2) {
              const int c2 = kKeep ? 1 - i2 : i2;
              if (!kKeep || c2 == 0) {
                tmem_ld32(tb + 64 * c2, *reinterpret_cast<uint32_t(*)[32]>(&s64[0]));
                tmem_ld32(tb + 64 * c2 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s64[32]));
                tmem_wait_ld();
                if (i2 == 1) {
                  // the last of S_g is in registers: the buffer can take S_{g+2}
                  tc_fence_before();
                  mbar_arrive(bar(B_SFREE + par));
                }
                if (kMasked && lim < 64 * (c2 + 1)) {
#pragma unroll
                  for (int j = 0; j < 64; ++j)
                    if (64 * c2 + j >= lim) s64[j] = __float_as_uint(-INFINITY);
                }
              }
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * c2 + cc;
                const uint32_t* sv = &s64[32 * cc];
                uint32_t w[4];
#pragma unroll
                for (int gg = 0; gg < 2; ++gg) {
                  const int q = 2 * c + gg;
                  const uint64_t bb = pack2(bias[q], bias[q]), l2 = pack2(lsc[q], lsc[q]);
                  float y[16];
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    const uint64_t x = fma2(
                        pack2(__uint_as_float(sv[16 * gg + 2 * e]), __uint_as_float(sv[16 * gg + 2 * e + 1])),
                        a2, bb);
                    y[2 * e] = ex2_approx(lo2(x));
                    y[2 * e + 1] = ex2_approx(hi2(x));
                    if constexpr (!kDirectP) acc[e & 1] = fma2(pack2(y[2 * e], y[2 * e + 1]), l2, acc[e & 1]);
                  }
                  float y8[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) y8[e] = y[e];
                  w[2 * gg] = cvt_e2m1x8(y8);
#pragma unroll
                  for (int e = 0; e < 8; ++e) y8[e] = y[8 + e];
                  w[2 * gg + 1] = cvt_e2m1x8(y8);
                  if constexpr (kDirectP)
                    rsum = fmaf(lsc[q], h2_total(e2m1x8_sum_h2(w[2 * gg]), e2m1x8_sum_h2(w[2 * gg + 1])), rsum);
                }
                *reinterpret_cast<uint4*>(prow + ((c ^ sw) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
            constexpr int kRowB = (D == 64) ? 16 * 128 : 16 * 32;  // bytes of one step's rows
            uint8_t* sfp = sm + L::oSFP + ps * L::SFPB + (D == 64 ? r : r % 32) * 16 + (r / 32) * 4;
            *reinterpret_cast<uint32_t*>(sfp) = __byte_perm(s2[0], s2[1], 0x5410);
            *reinterpret_cast<uint32_t*>(sfp + kRowB) = __byte_perm(s2[2], s2[3], 0x5410);
            const uint64_t acc2 = add2(acc[0], acc[1]);
            reinterpret_cast<float2*>(sm + L::oStat + (g % kEvRing) * 1024)[r] =
                make_float2(t, kDirectP ? rsum : lo2(acc2) + hi2(acc2));
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_PFULL + g % kEvRing));
            return true;
          };
          if (__any_sync(kFull, lim < kTileKV) ? !tile(std::true_type{}) : !tile(std::false_type{})) {
            ok = false;
            break;
          }
        }
        g0 += I.nkv;
      }
    }
    tc_fence_before();
    cta_bar_sync();
  } else {
    // -------------------------------------------------------- correction + epilogue
    regs_inc<Regs<D>::kCorr>();
    if (!skip) {
      const int r = threadIdx.x - 384;
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const float a = p.a;
      bool ok = true;
      int g = 0;
      for (int it = item0; ok && it < n_items; it += istep) {
        const Item I = item_at(p, it);
        uint64_t o2[D / 2];  // O row, two FP32 columns per register pair
#pragma unroll
        for (int d = 0; d < D / 2; ++d) o2[d] = 0ull;
        // m is the row's reference maximum: O and l are kept relative to it.
        // It moves only when a tile's maximum exceeds it by more than 8 / a
        // (a factor 2^8 on O), so most tiles skip the rescale of O; the result
        // is the same up to rounding, since O / l does not depend on m.
        float m = -INFINITY, l = 0.0f;
        for (int k = 0; k < I.nkv; ++k, ++g) {
          // the row stats of tile g are written before P_g is announced
          if (!(ok = waitw(bar(B_PFULL + g % kEvRing), (g / kEvRing) & 1, ctl))) break;
          const float2 st = reinterpret_cast<const float2*>(sm + L::oStat + (g % kEvRing) * 1024)[r];
          const bool up = (st.x - m) * a > 8.0f;
          const float mn = up ? st.x : m;
          const float alpha = up ? ex2_approx((m - mn) * a) : 1.0f;
          const float beta = ex2_approx((st.x - mn) * a);
          l = l * alpha + st.y * beta;
          const float w = beta * (kMx ? 1.0f / 6.0f : 1.0f / 2688.0f);
          m = mn;
          const bool keep = !__any_sync(kFull, up);  // no row of the warp moved its reference
          const uint64_t w2 = pack2(w, w), al2 = pack2(alpha, alpha);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int e = g * NH + h, pb = e % kPvBufs;
            if (!(ok = waitw(bar(B_PVDONE + e % kPvRing), (e / kPvRing) & 1, ctl))) break;
            tc_fence_after();
            // CW columns per wait (64 at D = 128, 32 at D = 64: measured)
            constexpr int CW = (D == 128) ? 64 : 32;
#pragma unroll
            for (int c = 0; c < D / CW; ++c) {
              uint32_t v[CW];
#pragma unroll
              for (int x = 0; x < CW / 32; ++x)
                tmem_ld32(tmem + kColPV + pb * D + CW * c + 32 * x + lane_base,
                          *reinterpret_cast<uint32_t(*)[32]>(&v[32 * x]));
              tmem_wait_ld();
              if (c == D / CW - 1) {
                // all of PV_e is in registers: its buffer is free
                tc_fence_before();
                mbar_arrive(bar(B_PVFREE + pb));
              }
              uint64_t* oc = &o2[(CW / 2) * c];
              if (keep) {
#pragma unroll
                for (int j = 0; j < CW / 2; ++j)
                  oc[j] = fma2(pack2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), w2, oc[j]);
              } else {
#pragma unroll
                for (int j = 0; j < CW / 2; ++j)
                  oc[j] = fma2(pack2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), w2,
                               mul2(oc[j], al2));
              }
            }
          }
          if (!ok) break;
        }
        const int gi = I.qt * kTileQ + r;
        if (ok && gi < p.N) {
          const float inv = 1.0f / l;
          // Dense [B,H,N,D] O (kDenseO) takes the plain row index; any other
          // layout its strides.  Two instantiations, because the general
          // address arithmetic in this spot measured 4-8% slower on the dense
          // case (the correction warpgroup's code is that tight).
          size_t row;
          if constexpr (kDenseO) {
            row = (static_cast<size_t>(I.bh) * p.N + gi) * D;
          } else {
            const unsigned b = static_cast<unsigned>(I.bh) / static_cast<unsigned>(p.H);
            const unsigned h = static_cast<unsigned>(I.bh) - b * static_cast<unsigned>(p.H);
            row = static_cast<size_t>(b) * static_cast<size_t>(p.os.b) +
                  static_cast<size_t>(h) * static_cast<size_t>(p.os.h) +
                  static_cast<size_t>(gi) * static_cast<size_t>(p.os.n);
          }
          uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + row);
#if SAGE_FP4_DEBUG_BOUNDS
          if (!in_bounds(p.ext, static_cast<long long>(row), D, p.ext.o)) orow = nullptr;
#pragma unroll
          for (int c = 0; c < D / 8 && orow; ++c) {
#else
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
#endif
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 h2 =
                  __floats2bfloat162_rn(lo2(o2[c * 4 + e]) * inv, hi2(o2[c * 4 + e]) * inv);
              w4[e] = *reinterpret_cast<uint32_t*>(&h2);
            }
            orow[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
    }
    tc_fence_before();
    cta_bar_sync();
  }
}

int num_sms_attn() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

template <int D, bool kDenseO, bool kMx, bool kDirectP = false>
cudaError_t launch_attn_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const AttnParams& p, cudaStream_t st) {
  static int configured_mask = 0;  // one bit per device ordinal (< 32)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 32 || !(configured_mask & (1 << dev))) {
    // The warpgroups' setmaxnreg budgets add up to exactly 128 registers per
    // thread at launch; with any other launch allocation the increases would
    // never be granted, so refuse to launch.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, attn_fwd_kernel<D, kDenseO, kMx, kDirectP>);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != 65536 / kThreads) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(attn_fwd_kernel<D, kDenseO, kMx, kDirectP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<D>::kAlloc);
    if (e != cudaSuccess) return e;
    if (dev < 32) configured_mask |= (1 << dev);
  }
  // persistent: one CTA per SM (it owns all of the SM's tensor memory), each
  // taking items blockIdx.x, blockIdx.x + gridDim.x, ...
  const long long items = static_cast<long long>(p.BH) * p.n_qt;
  const long long sms = num_sms_attn();
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  attn_fwd_kernel<D, kDenseO, kMx, kDirectP><<<grid, kThreads, Smem<D>::kAlloc, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const AttnParams& p, int D, cudaStream_t st) {
  const Strides dense = contiguous_bhnd(p.H, p.N, D);
  const bool dense_o = p.os.b == dense.b && p.os.h == dense.h && p.os.n == dense.n;
  if (p.mx == 2) {
    // Direct-P (MXFP4): dense O only (the API checks it)
    if (!dense_o) return cudaErrorInvalidValue;
    return D == 128 ? launch_attn_d<128, true, true, true>(tq, tk, tv, p, st)
                    : launch_attn_d<64, true, true, true>(tq, tk, tv, p, st);
  }
  if (p.mx) {
    if (D == 128)
      return dense_o ? launch_attn_d<128, true, true>(tq, tk, tv, p, st)
                     : launch_attn_d<128, false, true>(tq, tk, tv, p, st);
    return dense_o ? launch_attn_d<64, true, true>(tq, tk, tv, p, st)
                   : launch_attn_d<64, false, true>(tq, tk, tv, p, st);
  }
  if (D == 128)
    return dense_o ? launch_attn_d<128, true, false>(tq, tk, tv, p, st)
                   : launch_attn_d<128, false, false>(tq, tk, tv, p, st);
  return dense_o ? launch_attn_d<64, true, false>(tq, tk, tv, p, st)
                 : launch_attn_d<64, false, false>(tq, tk, tv, p, st);
}

}  // namespace sagefp4

// layout.cuh -- sizes and byte layouts of the quantized operands (see
// include/sage_fp4.h) and of the attention kernel's shared/tensor memory.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace sagefp4 {

constexpr int kTileQ = 128;   // query rows per attention tile (one CTA)
constexpr int kTileKV = 128;  // keys per KV tile (the level-1 normalisation unit)
constexpr int kGroup = 16;    // NVFP4 microscaling group

__host__ __device__ constexpr int round_up_int(int x, int m) { return (x + m - 1) / m * m; }
__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte offset of the scale of (row r, group g) in the 128x4 block layout of an
// operand whose contraction axis holds `groups` groups (a multiple of 4).
__host__ __device__ inline size_t sf_offset(int r, int g, int groups) {
  return (static_cast<size_t>(r / 128) * (groups / 4) + g / 4) * 512 + (r % 32) * 16 +
         ((r % 128) / 32) * 4 + (g % 4);
}

// Per-(b,h) sizes of the quantized operands.
struct OperandSizes {
  size_t q_codes, q_scales;    // per tensor Q or K
  size_t vt_codes, vt_scales;  // V^T
};

__host__ __device__ inline OperandSizes operand_sizes(int N, int D) {
  const int Np = round_up_int(N, 128);
  OperandSizes s;
  s.q_codes = static_cast<size_t>(Np) * D / 2;
  s.q_scales = static_cast<size_t>(Np) * D / 16;
  s.vt_codes = static_cast<size_t>(D) * Np / 2;
  s.vt_scales = static_cast<size_t>(128) * Np / 16;
  return s;
}

}  // namespace sagefp4

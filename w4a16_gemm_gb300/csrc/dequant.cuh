// dequant.cuh -- register dequantization of one packed 32-bit word.
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "tmw4_device.cuh"

namespace tmw4 {

// Eight codes of one word (value e at nibble NIBBLE_POS[e], i.e. word order
// e7 e5 e3 e1 e6 e4 e2 e0 -- pith.science review, Figures 23/24) become four
// packed 16-bit pairs {w0,w1}, {w2,w3}, {w4,w5}, {w6,w7} (low half = even
// element), with w = T(s * (q - z)):
//   mask 0x000F000F after a shift by 4i isolates the pair (e_2i, e_2i+1);
//   OR-ing the exponent magic gives MAGIC + q exactly; subtracting the
//   duplicated (MAGIC + z) is exact; the multiply by the duplicated scale is
//   the single round-to-nearest-even.
// zm2 = (MAGIC + z) in both halves, s2 = scale in both halves.
template <bool BF16>
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t zm2, uint32_t s2,
                                             uint32_t (&out)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t x = ((w >> (4 * i)) & 0x000F000Fu) | Magic<BF16>::pair;
    if constexpr (BF16) {
      out[i] = mul_rn_bf16x2(sub_rn_bf16x2(x, zm2), s2);
    } else {
      out[i] = mul_rn_f16x2(sub_rn_f16x2(x, zm2), s2);
    }
  }
}

// (MAGIC + z) duplicated into both 16-bit halves.
template <bool BF16>
__device__ __forceinline__ uint32_t zero_magic2(uint32_t z) {
  const uint32_t h = Magic<BF16>::one + z;
  return h | (h << 16);
}

__device__ __forceinline__ uint32_t dup16(uint32_t h) { return (h & 0xFFFFu) | (h << 16); }

// Zero point of column n in group g from the tile-major nibble array; 8 for
// the symmetric format (zeros == nullptr).
__device__ __forceinline__ uint32_t zero_of(const uint8_t *zeros, int g, int n, int G_rows) {
  if (zeros == nullptr) return 8u;
  return (static_cast<uint32_t>(zeros[zero_byte(g, n, G_rows)]) >> ((n & 1) * 4)) & 0xFu;
}

}  // namespace tmw4

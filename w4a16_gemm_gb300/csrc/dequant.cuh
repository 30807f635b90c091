// dequant.cuh -- register dequantization of one packed 32-bit word.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "tmw4_device.cuh"

namespace tmw4 {

// Eight codes of one word (value e at nibble NIBBLE_POS[e], i.e. word order
// e7 e5 e3 e1 e6 e4 e2 e0 -- pith.science review, Figures 23/24) become four
// packed 16-bit pairs {w0,w1}, {w2,w3}, {w4,w5}, {w6,w7} (low half = even
// element), with w = T(s * (q - z)) rounded once to nearest even.
//
// fp16: nibble pairs (e0,e1) and (e4,e5) sit in the low nibble of each
// half-word (directly, and after one shift by 8); OR-ing 0x6400 gives
// 1024 + q exactly and subtracting the duplicated 1024 + z is exact.  Pairs
// (e2,e3) and (e6,e7) sit one nibble higher: OR-ing 0x6400 gives 1024 + 16q
// exactly, and one fused x * (1/16) - (64 + z) yields q - z exactly (the
// product is exact, so the single rounding of the FMA is exact too).  The
// multiply by the scale is the only rounding of w.  bf16 (7 mantissa bits)
// has no room for the higher nibble, so every pair is shifted down first.
// zm2 = (MAGIC + z) in both halves, s2 = scale in both halves.
template <bool BF16>
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t zm2, uint32_t s2,
                                             uint32_t (&out)[4]) {
  if constexpr (BF16) {
    const __nv_bfloat162 z = *reinterpret_cast<const __nv_bfloat162 *>(&zm2);
    const __nv_bfloat162 s = *reinterpret_cast<const __nv_bfloat162 *>(&s2);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t x = ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
      __nv_bfloat162 d = __hmul2(__hsub2(*reinterpret_cast<__nv_bfloat162 *>(&x), z), s);
      out[i] = *reinterpret_cast<uint32_t *>(&d);
    }
  } else {
    const __half2 z = *reinterpret_cast<const __half2 *>(&zm2);
    const __half2 s = *reinterpret_cast<const __half2 *>(&s2);
    // -(64 + z) = 960 - (1024 + z), exact
    const __half2 z16 = __hsub2(__float2half2_rn(960.0f), z);
    const __half2 sixteenth = __float2half2_rn(0.0625f);
    const uint32_t hi = w >> 8;
    uint32_t x0 = (w & 0x000F000Fu) | 0x64006400u;
    uint32_t x1 = (w & 0x00F000F0u) | 0x64006400u;
    uint32_t x2 = (hi & 0x000F000Fu) | 0x64006400u;
    uint32_t x3 = (hi & 0x00F000F0u) | 0x64006400u;
    const __half2 d0 = __hsub2(*reinterpret_cast<__half2 *>(&x0), z);
    const __half2 d1 = __hfma2(*reinterpret_cast<__half2 *>(&x1), sixteenth, z16);
    const __half2 d2 = __hsub2(*reinterpret_cast<__half2 *>(&x2), z);
    const __half2 d3 = __hfma2(*reinterpret_cast<__half2 *>(&x3), sixteenth, z16);
    __half2 r0 = __hmul2(d0, s), r1 = __hmul2(d1, s), r2 = __hmul2(d2, s), r3 = __hmul2(d3, s);
    out[0] = *reinterpret_cast<uint32_t *>(&r0);
    out[1] = *reinterpret_cast<uint32_t *>(&r1);
    out[2] = *reinterpret_cast<uint32_t *>(&r2);
    out[3] = *reinterpret_cast<uint32_t *>(&r3);
  }
}

// (MAGIC + z) duplicated into both 16-bit halves.
template <bool BF16>
__device__ __forceinline__ uint32_t zero_magic2(uint32_t z) {
  // one integer multiply-add (FMA pipe) instead of three logic ops
  return z * 0x00010001u + Magic<BF16>::pair;
}

__device__ __forceinline__ uint32_t dup16(uint32_t h) { return (h & 0xFFFFu) * 0x00010001u; }

// 8-bit codes.  Four codes of one word (K order k..k+3, byte i = K k+i) become
// two packed 16-bit pairs {w0,w1}, {w2,w3} with w = T(s * v), one rounding:
//   int8 (v = q - z, q and z in 0..255):
//     fp16: a byte permute places each code under the exponent magic 0x6400
//           (1024 + q, exact for q <= 255); the subtract of 1024 + z is exact
//           (|q - z| <= 255); the multiply by the scale is the one rounding.
//     bf16: 7 mantissa bits cannot hold 128 + q for q >= 128, so each code
//           goes through fp32: 2^23 + q (exact), minus 2^23 + z (exact), times
//           s (exact: at most 17 significant bits), one rounding to bf16.
//   FP8 E4M3 (v = e4m3(q)): exact conversion to fp16 (cvt.rn.f16x2.e4m3x2),
//     then fp16: one multiply; bf16: widened to fp32 (exact), times s
//     (exact: at most 12 significant bits), one rounding to bf16.
// zm2 = (1024 + z) in both fp16 halves (int8, fp16), z8 = z (int8, bf16),
// s2 = the scale in both halves, sf = the scale in fp32.
template <bool BF16>
__device__ __forceinline__ void dequant_word8(uint32_t w, bool fp8, uint32_t zm2, uint32_t z8, uint32_t s2,
                                              float sf, uint32_t (&out)[2]) {
  if (fp8) {
    uint32_t h0, h1;   // fp16 pairs of bytes (0,1) and (2,3)
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h0), "=r"(h1)
        : "r"(w));
    if constexpr (BF16) {
      const uint32_t h[2] = {h0, h1};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const __half2 v = *reinterpret_cast<const __half2 *>(&h[i]);
        const float2 f = __half22float2(v);
        const __nv_bfloat162 r = __floats2bfloat162_rn(f.x * sf, f.y * sf);
        out[i] = *reinterpret_cast<const uint32_t *>(&r);
      }
    } else {
      const __half2 s = *reinterpret_cast<const __half2 *>(&s2);
      const __half2 r0 = __hmul2(*reinterpret_cast<const __half2 *>(&h0), s);
      const __half2 r1 = __hmul2(*reinterpret_cast<const __half2 *>(&h1), s);
      out[0] = *reinterpret_cast<const uint32_t *>(&r0);
      out[1] = *reinterpret_cast<const uint32_t *>(&r1);
    }
    return;
  }
  if constexpr (BF16) {
    const float zf = __uint_as_float(0x4B000000u | z8);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float a = (__uint_as_float(0x4B000000u | ((w >> (16 * i)) & 0xFFu)) - zf) * sf;
      const float b = (__uint_as_float(0x4B000000u | ((w >> (16 * i + 8)) & 0xFFu)) - zf) * sf;
      const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
      out[i] = *reinterpret_cast<const uint32_t *>(&r);
    }
  } else {
    const __half2 z = *reinterpret_cast<const __half2 *>(&zm2);
    const __half2 s = *reinterpret_cast<const __half2 *>(&s2);
    const uint32_t x0 = __byte_perm(w, 0x6464u, 0x5140u);   // {0x64, byte1, 0x64, byte0} -> (1024+q0, 1024+q1)
    const uint32_t x1 = __byte_perm(w, 0x6464u, 0x5342u);
    const __half2 r0 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&x0), z), s);
    const __half2 r1 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&x1), z), s);
    out[0] = *reinterpret_cast<const uint32_t *>(&r0);
    out[1] = *reinterpret_cast<const uint32_t *>(&r1);
  }
}

// 8-bit zero point of column n in group g (tile-major bytes); 128 when there
// is none (symmetric int8, and FP8, whose path ignores it).
__device__ __forceinline__ uint32_t zero8_of(const uint8_t *zeros, int g, int n, int G_rows) {
  if (zeros == nullptr) return 128u;
  return zeros[(static_cast<size_t>(n >> 7) * G_rows + g) * TILE_N + (n & 127)];
}

// Zero point of column n in group g from the tile-major nibble array; 8 for
// the symmetric format (zeros == nullptr).
__device__ __forceinline__ uint32_t zero_of(const uint8_t *zeros, int g, int n, int G_rows) {
  if (zeros == nullptr) return 8u;
  return (static_cast<uint32_t>(zeros[zero_byte(g, n, G_rows)]) >> ((n & 1) * 4)) & 0xFu;
}

}  // namespace tmw4

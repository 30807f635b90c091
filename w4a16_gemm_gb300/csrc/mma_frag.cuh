// mma_frag.cuh -- register-operand tensor-core pieces shared by the
// kernels that multiply dequantized weights with mma.sync m16n8k16: exact
// (q - z) dequantization into 16-bit pairs, the MMA itself, and fp32 helpers.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tmw4 {

// Eight codes of one packed word (value e at nibble (0,4,1,5,2,6,3,7)[e]) ->
// four 16-bit pairs (q_e - z), exact: {e0,e1}, {e2,e3}, {e4,e5}, {e6,e7},
// the even element in the low half.
//   fp16: OR-ing 0x6400 into a nibble in the low mantissa bits gives 1024 + q
//         exactly; one nibble higher it gives 1024 + 16q exactly.  The first
//         form minus (1024 + z) and the second form times 1/16 minus (64 + z)
//         (a fused multiply-add whose exact result is a small integer) are
//         both exact.  One shift, four lop3 (mask and OR in one), two subtracts
//         and two fused multiply-adds per word.
//   bf16: only 7 mantissa bits, so each pair is shifted to the low nibble
//         first; 0x4300 gives 128 + q exactly, minus (128 + z) is exact.
// zm = (MAGIC + z) in both halves; z16 = -(64 + z) in both halves (fp16 only).
// Written in PTX so that each mask-and-OR is one lop3 (the C++ form of the
// same expression compiled to twice as many logic instructions).
template <bool BF16>
__device__ __forceinline__ void codes_minus_zero(uint32_t w, uint32_t zm, uint32_t z16,
                                                 uint32_t (&out)[4]) {
  if constexpr (BF16) {
    asm("{\n\t.reg .b32 s1, s2, s3, x0, x1, x2, x3;\n\t"
        "shr.b32 s1, %4, 4;\n\t"
        "shr.b32 s2, %4, 8;\n\t"
        "shr.b32 s3, %4, 12;\n\t"
        "lop3.b32 x0, %4, 0x000F000F, 0x43004300, 0xEA;\n\t"
        "lop3.b32 x1, s1, 0x000F000F, 0x43004300, 0xEA;\n\t"
        "lop3.b32 x2, s2, 0x000F000F, 0x43004300, 0xEA;\n\t"
        "lop3.b32 x3, s3, 0x000F000F, 0x43004300, 0xEA;\n\t"
        "sub.rn.bf16x2 %0, x0, %5;\n\t"
        "sub.rn.bf16x2 %1, x1, %5;\n\t"
        "sub.rn.bf16x2 %2, x2, %5;\n\t"
        "sub.rn.bf16x2 %3, x3, %5;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(w), "r"(zm));
    (void)z16;
  } else {
    asm("{\n\t.reg .b32 hi, x0, x1, x2, x3;\n\t"
        "shr.b32 hi, %4, 8;\n\t"
        "lop3.b32 x0, %4, 0x000F000F, 0x64006400, 0xEA;\n\t"
        "lop3.b32 x1, %4, 0x00F000F0, 0x64006400, 0xEA;\n\t"
        "lop3.b32 x2, hi, 0x000F000F, 0x64006400, 0xEA;\n\t"
        "lop3.b32 x3, hi, 0x00F000F0, 0x64006400, 0xEA;\n\t"
        "sub.rn.f16x2 %0, x0, %5;\n\t"
        "fma.rn.f16x2 %1, x1, %7, %6;\n\t"
        "sub.rn.f16x2 %2, x2, %5;\n\t"
        "fma.rn.f16x2 %3, x3, %7, %6;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(w), "r"(zm), "r"(z16), "r"(0x2C002C00u));   // 0x2C00 = 1/16
  }
}

// Four 8-bit codes of one word (byte e = value e) -> two exact 16-bit pairs
// {e0,e1}, {e2,e3} of (q - z), or of e4m3(q) for FP8 codes (no zero point).
//   fp16 int8: a byte permute places each code under the exponent magic
//              0x6400 (1024 + q, exact for q <= 255); minus (1024 + z) is exact.
//   bf16 int8: 2^23 + q in fp32 minus 2^23 + z (exact), converted to bf16
//              exactly (|q - z| <= 255 has at most 8 significant bits).
//   FP8: the hardware E4M3 -> f16x2 conversion is exact; for bf16 each half
//        is widened to fp32 and narrowed to bf16, both exact (E4M3 values
//        have 4 significant bits and exponents inside bf16's range).
// zm = (1024 + z) in both fp16 halves; zf = 2^23 + z as fp32.
template <bool BF16>
__device__ __forceinline__ void codes8_minus_zero(uint32_t w, uint32_t zm, float zf, bool fp8, uint32_t &p01,
                                                  uint32_t &p23) {
  if (fp8) {
    uint32_t h0, h1;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h0), "=r"(h1)
        : "r"(w));
    if constexpr (BF16) {
      const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&h0));
      const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&h1));
      const __nv_bfloat162 b0 = __floats2bfloat162_rn(f0.x, f0.y), b1 = __floats2bfloat162_rn(f1.x, f1.y);
      p01 = *reinterpret_cast<const uint32_t *>(&b0);
      p23 = *reinterpret_cast<const uint32_t *>(&b1);
    } else {
      p01 = h0;
      p23 = h1;
    }
    return;
  }
  if constexpr (BF16) {
    (void)zm;
    const float q0 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u)) - zf;
    const float q1 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541u)) - zf;
    const float q2 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542u)) - zf;
    const float q3 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543u)) - zf;
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(q0, q1), b1 = __floats2bfloat162_rn(q2, q3);
    p01 = *reinterpret_cast<const uint32_t *>(&b0);
    p23 = *reinterpret_cast<const uint32_t *>(&b1);
  } else {
    (void)zf;
    asm("{\n\t.reg .b32 x0, x1;\n\t"
        "prmt.b32 x0, %2, 0x64646464, 0x4140;\n\t"
        "prmt.b32 x1, %2, 0x64646464, 0x4342;\n\t"
        "sub.rn.f16x2 %0, x0, %3;\n\t"
        "sub.rn.f16x2 %1, x1, %3;\n\t}"
        : "=r"(p01), "=r"(p23)
        : "r"(w), "r"(zm));
  }
}

// d.xy += s.xy * a.xy, two fp32 lanes in one instruction.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float s0, float s1, float a0, float a1) {
  asm("{\n\t.reg .b64 d, s, a;\n\t"
      "mov.b64 d, {%0, %1};\n\t"
      "mov.b64 s, {%2, %3};\n\t"
      "mov.b64 a, {%4, %5};\n\t"
      "fma.rn.f32x2 d, s, a, d;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(s0), "f"(s1), "f"(a0), "f"(a1));
}

// d += A(16x16, row) * B(16x8, col), fp32 accumulate.
template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

template <bool BF16>
__device__ __forceinline__ float bits16_to_f32(uint32_t h) {
  return BF16 ? __uint_as_float(h << 16) : __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

template <bool BF16>
__device__ __forceinline__ uint16_t f32_to_bits16(float x) {
  if constexpr (BF16) {
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&b);
  } else {
    __half h = __float2half_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
  }
}


}  // namespace tmw4

// tmw4_device.cuh -- device-side constants and the int4 -> 16-bit dequant
// step shared by the kernels of this library.
#pragma once

#include <cstdint>

namespace tmw4 {

// Bits of the per-device error word (read and cleared by tm_poll_error).
constexpr unsigned int TM_DEVERR_TIMEOUT = 1u;   // a bounded wait gave up
constexpr unsigned int TM_DEVERR_BAD_CODE = 2u;  // a code byte above 15 was packed

// Geometry of the packed weight (see include/tmw4.h).
constexpr int ATOM_K = 64;
constexpr int ATOM_N = 64;
constexpr int ATOM_BYTES = ATOM_K * ATOM_N / 2;  // 2048

// Exponent "magic" that turns a 4-bit code c placed in the low mantissa bits
// into the exact value MAGIC + c: 1024 + c for fp16 (0x6400), 128 + c for
// bf16 (0x4300).  Subtracting (MAGIC + z) is exact, so the following multiply
// by the scale is the only rounding: w = T(s * (q - z)), round to nearest
// even (runtime I2F conversion and scaling: TurboMind paper, pith.science
// review, Figure 6).
template <bool BF16>
struct Magic {
  static constexpr uint32_t pair = BF16 ? 0x43004300u : 0x64006400u;
  static constexpr uint32_t one = BF16 ? 0x4300u : 0x6400u;
};

}  // namespace tmw4

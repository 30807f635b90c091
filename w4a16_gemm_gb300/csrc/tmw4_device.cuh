// tmw4_device.cuh -- device-side constants and the int4 -> 16-bit dequant
// step shared by the kernels of this library.
#pragma once

#include <cstdint>

namespace tmw4 {

// Bits of the per-device error word (read and cleared by tm_poll_error).
constexpr unsigned int TM_DEVERR_TIMEOUT = 1u;   // a bounded wait gave up
constexpr unsigned int TM_DEVERR_BAD_CODE = 2u;  // a code byte above 15 was packed
constexpr int TM_ERR_WORDS = 8;                  // error word + where the first wait gave up

// Wait sites recorded when a bounded wait gives up.
enum WaitSite : unsigned {
  SITE_PRODUCER_EMPTY = 1,
  SITE_MMA_FULL = 2,
  SITE_MMA_AFULL = 3,
  SITE_DQ_FULL = 4,
  SITE_DQ_AEMPTY = 5,
  SITE_EPI_ACCUM = 6,
  SITE_DRAIN_TMA = 7,
  SITE_DRAIN_MMA = 8,
  SITE_SELFTEST = 9
};

// Geometry of the packed weight (see include/tmw4.h): 128-column tiles,
// each tile's 64-K blocks contiguous (4096 bytes = two 2048-byte atoms of
// 64 columns); scales [N/128][K/G][128], zeros [N/128][K/G][64 bytes].
constexpr int ATOM_K = 64;
constexpr int ATOM_N = 64;
constexpr int ATOM_BYTES = ATOM_K * ATOM_N / 2;  // 2048
constexpr int TILE_N = 128;
constexpr int BLOCK_BYTES = 2 * ATOM_BYTES;      // one tile x one 64-K block

// Byte offset of atom (kb, na) (na = 64-column index) in the packed stream.
__host__ __device__ __forceinline__ size_t atom_offset(int kb, int na, int KB) {
  return (static_cast<size_t>(na >> 1) * KB + kb) * BLOCK_BYTES +
         static_cast<size_t>(na & 1) * ATOM_BYTES;
}
// Index of scale (g, n) in the tile-major scale array (G_rows = K/G).
__host__ __device__ __forceinline__ size_t scale_index(int g, int n, int G_rows) {
  return (static_cast<size_t>(n >> 7) * G_rows + g) * TILE_N + (n & 127);
}
// Byte holding zero (g, n) in the tile-major nibble array (odd n: high nibble).
__host__ __device__ __forceinline__ size_t zero_byte(int g, int n, int G_rows) {
  return (static_cast<size_t>(n >> 7) * G_rows + g) * (TILE_N / 2) + ((n & 127) >> 1);
}

// Stream-K partition of U work units over a persistent grid of G CTAs: CTA c
// owns units [unit_begin(c), unit_begin(c + 1)).
__host__ __device__ __forceinline__ long long unit_begin(long long c, long long U, long long G) {
  return c * U / G;
}
// The CTA whose range holds unit u.
__host__ __device__ __forceinline__ int cta_of_unit(long long u, long long U, long long G) {
  long long c = u * G / U;
  while (c + 1 < G && unit_begin(c + 1, U, G) <= u) ++c;
  while (c > 0 && unit_begin(c, U, G) > u) --c;
  return static_cast<int>(c);
}

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

// Debug timeline: with TMW4_TRACE defined, kernels record clock64() stamps of
// pipeline events of CTA (0,0,0) into GemmArgs::trace[slot * 256 + idx].
#ifdef TMW4_TRACE
#define TMW4_STAMP(slot, idx)                                                              \
  do {                                                                                     \
    if (p.trace != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&     \
        (idx) < 256)                                                                       \
      p.trace[(slot) * 256 + (idx)] = clock64();                                           \
  } while (0)
#else
#define TMW4_STAMP(slot, idx) \
  do {                        \
  } while (0)
#endif

// pack.cu -- offline repack of int4 codes into the library's packed layout,
// nibble-packing of zero points, and the dequant-only kernel.
//
// Repack follows the pages' offline packing (TurboMind paper, pith.science
// review, Figures 6/7: load a tile, place each thread's eight values, permute
// them into MMA order and store fragments in the order the runtime loads
// them).  Here one CTA moves one 64x64 atom: a coalesced 4 KB load of codes
// into shared memory, then 512 packed words written contiguously.
#include <cstdint>
#include <cuda_runtime.h>

#include "dequant.cuh"
#include "kernels.h"
#include "tmw4_device.cuh"

namespace tmw4 {

// NIBBLE_POS of the layout: value e of a word sits at nibble kNibPos[e].
__device__ __constant__ int kNibPos[8] = {0, 4, 1, 5, 2, 6, 3, 7};

// Column offset within a group of eight held by nibble i of an AWQ-packed
// 32-bit word (the AWQ "GEMM" layout interleaves even and odd columns).
__device__ __constant__ int kAwqCol[8] = {0, 2, 4, 6, 1, 3, 5, 7};

// Source layouts of the codes (SrcLayout):
//   U8    q [K][N] bytes, one code per byte;
//   AWQ   int32 [K][N/8]: word (k, j) holds columns 8j + kAwqCol[i] of row k
//         in nibble i;
//   GPTQ  int32 [K/8][N]: word (r, n) holds rows 8r + i of column n in
//         nibble i.
template <int SRC>
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t *__restrict__ q,
                                                     uint8_t *__restrict__ qw, int K, int N,
                                                     unsigned int *err) {
  __shared__ uint8_t tile[ATOM_K][ATOM_N + 4];
  const int na = blockIdx.x, kb = blockIdx.y, t = threadIdx.x;
  const int k0 = kb * ATOM_K, n0 = na * ATOM_N;
  if constexpr (SRC == SRC_U8) {
    // 64 rows x 64 bytes, 16 bytes per thread
    const int row = t >> 2, col = (t & 3) * 16;
    const uint4 v = *reinterpret_cast<const uint4 *>(q + static_cast<size_t>(k0 + row) * N + n0 + col);
    if (((v.x | v.y | v.z | v.w) & 0xF0F0F0F0u) != 0u) atomicOr(err, TM_DEVERR_BAD_CODE);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int b = 0; b < 4; ++b) tile[row][col + 4 * i + b] = (w[i] >> (8 * b)) & 0xFu;
    }
  } else if constexpr (SRC == SRC_AWQ) {
    // 64 rows x 8 words; two words (16 columns) per thread
    const uint32_t *src = reinterpret_cast<const uint32_t *>(q);
    const int row = t >> 2, j0 = (t & 3) * 2;
    const uint2 v = *reinterpret_cast<const uint2 *>(src + static_cast<size_t>(k0 + row) * (N / 8) + n0 / 8 + j0);
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
      for (int i = 0; i < 8; ++i) tile[row][8 * (j0 + jj) + kAwqCol[i]] = (w[jj] >> (4 * i)) & 0xFu;
  } else {
    // 8 word rows (64 K) x 64 columns; two words (two columns) per thread
    const uint32_t *src = reinterpret_cast<const uint32_t *>(q);
    const int r = t >> 5, col = (t & 31) * 2;
    const uint2 v = *reinterpret_cast<const uint2 *>(src + static_cast<size_t>(k0 / 8 + r) * N + n0 + col);
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int i = 0; i < 8; ++i) tile[8 * r + i][col + c] = (w[c] >> (4 * i)) & 0xFu;
  }
  __syncwarp();   // rejoin lanes that took the error branch before the CTA barrier
  __syncthreads();
  uint32_t *out = reinterpret_cast<uint32_t *>(qw + atom_offset(kb, na, K / ATOM_K));
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int widx = t + 256 * r;
    const int h = widx >> 8, nl = (widx & 255) >> 2, j = widx & 3;
    const int o = 4 * h + j;
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) word |= static_cast<uint32_t>(tile[8 * o + e][nl]) << (4 * kNibPos[e]);
    out[widx] = word;
  }
}

// zeros -> tile-major nibbles; one thread per output byte.  Packed group
// row g takes source row g / rep (a coarser group repeated rep times).
// Sources: U8 [K/G][N] bytes; AWQ int32 [K/G][N/8] in the AWQ column order;
// GPTQ int32 [K/G][N/8] with column 8c + i in nibble i.  `offset` is added
// to every zero (GPTQ files store zero - 1); a result above 15 is a bad code.
template <int SRC>
__global__ void pack_zeros_kernel(const uint8_t *__restrict__ z, uint8_t *__restrict__ zp,
                                  int rows, int N, int rep, int offset, unsigned int *err) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t total = static_cast<size_t>(rows) * (N / 2);
  if (i >= total) return;
  const size_t g = i / (N / 2), c = i % (N / 2);
  const size_t gs = g / rep;
  const int n = static_cast<int>(2 * c);
  uint32_t zz[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int nn = n + h;
    if constexpr (SRC == SRC_U8) {
      zz[h] = z[gs * N + nn];
    } else {
      const uint32_t w = reinterpret_cast<const uint32_t *>(z)[gs * (N / 8) + nn / 8];
      const int pos = SRC == SRC_AWQ ? (nn % 8 % 2 == 0 ? (nn % 8) / 2 : 4 + (nn % 8) / 2) : nn % 8;
      zz[h] = ((w >> (4 * pos)) & 0xFu) + static_cast<uint32_t>(offset);
    }
  }
  if ((zz[0] | zz[1]) > 15u) atomicOr(err, TM_DEVERR_BAD_CODE);
  zp[zero_byte(static_cast<int>(g), n, rows)] = static_cast<uint8_t>((zz[0] & 0xFu) | ((zz[1] & 0xFu) << 4));
}

// scales [K/G][N] -> tile-major [N/128][rows][128]; one thread per packed
// scale, row g from source row g / rep.
__global__ void pack_scales_kernel(const uint16_t *__restrict__ s, uint16_t *__restrict__ sp,
                                   int rows, int N, int rep) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<size_t>(rows) * N) return;
  const int g = static_cast<int>(i / N), n = static_cast<int>(i % N);
  sp[scale_index(g, n, rows)] = s[static_cast<size_t>(g / rep) * N + n];
}

// One thread per 16-byte chunk: 32 consecutive K values of one column.
template <bool BF16>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ qw,
                                                      const uint16_t *__restrict__ scales,
                                                      const uint8_t *__restrict__ zeros,
                                                      uint16_t *__restrict__ out, int K, int N,
                                                      int group) {
  const size_t c = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nchunks = static_cast<size_t>(K) * N / 32;
  if (c >= nchunks) return;
  const int KB = K / ATOM_K, G_rows = K / group;
  const size_t block = c >> 8;                     // 4096-byte tile block
  const int nt = static_cast<int>(block / KB), kb = static_cast<int>(block % KB);
  const int inblk = static_cast<int>(c & 255), a = inblk >> 7, h = (inblk >> 6) & 1, nl = inblk & 63;
  const int k0 = kb * ATOM_K + 32 * h, n = nt * TILE_N + a * ATOM_N + nl;
  const int g = k0 / group;
  const uint32_t s2 = dup16(scales[scale_index(g, n, G_rows)]);
  const uint32_t zm2 = zero_magic2<BF16>(zero_of(zeros, g, n, G_rows));
  const uint4 v = *reinterpret_cast<const uint4 *>(qw + c * 16);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t d[4];
    dequant_word<BF16>(w[j], zm2, s2, d);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const size_t k = static_cast<size_t>(k0 + 8 * j + 2 * i);
      out[k * N + n] = static_cast<uint16_t>(d[i] & 0xFFFFu);
      out[(k + 1) * N + n] = static_cast<uint16_t>(d[i] >> 16);
    }
  }
}

// ------------------------------------------------------------ 8-bit weights
// Packed 8-bit layout: 128-column tiles, 64-K blocks of 8192 bytes at
// (nt * K/64 + kb) * 8192; inside a block, 16-byte chunk kq * 128 + c holds
// the 16 consecutive K values 64 kb + 16 kq + (0..15) of column 128 nt + c.
// One thread per chunk; a warp's threads take consecutive columns, so each
// of the 16 rows it reads is 32 contiguous bytes.
__global__ void __launch_bounds__(256) repack8_kernel(const uint8_t *__restrict__ q, uint8_t *__restrict__ qw,
                                                      int K, int N) {
  const size_t c = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= static_cast<size_t>(K) * N / 16) return;
  const int KB = K / ATOM_K;
  const size_t block = c >> 9;
  const int inblk = static_cast<int>(c & 511), kq = inblk >> 7, col = inblk & 127;
  const int nt = static_cast<int>(block / KB), kb = static_cast<int>(block % KB);
  const int k0 = kb * ATOM_K + 16 * kq, n = nt * TILE_N + col;
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < 16; ++e) w[e >> 2] |= static_cast<uint32_t>(q[static_cast<size_t>(k0 + e) * N + n]) << (8 * (e & 3));
  *reinterpret_cast<uint4 *>(qw + c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

// 8-bit zeros [K/G][N] bytes -> tile-major [N/128][rows][128] bytes; packed
// row g from source row g / rep.
__global__ void pack_zeros8_kernel(const uint8_t *__restrict__ z, uint8_t *__restrict__ zp, int rows, int N,
                                   int rep) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<size_t>(rows) * N) return;
  const int g = static_cast<int>(i / N), n = static_cast<int>(i % N);
  zp[(static_cast<size_t>(n >> 7) * rows + g) * TILE_N + (n & 127)] = z[static_cast<size_t>(g / rep) * N + n];
}

// Dequant-only for 8-bit weights; one thread per 16-byte chunk.
template <bool BF16>
__global__ void __launch_bounds__(256) dequant8_kernel(const uint8_t *__restrict__ qw,
                                                       const uint16_t *__restrict__ scales,
                                                       const uint8_t *__restrict__ zeros, int fp8,
                                                       uint16_t *__restrict__ out, int K, int N, int group) {
  const size_t c = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= static_cast<size_t>(K) * N / 16) return;
  const int KB = K / ATOM_K, G_rows = K / group;
  const size_t block = c >> 9;
  const int inblk = static_cast<int>(c & 511), kq = inblk >> 7, col = inblk & 127;
  const int nt = static_cast<int>(block / KB), kb = static_cast<int>(block % KB);
  const int k0 = kb * ATOM_K + 16 * kq, n = nt * TILE_N + col;
  const int g = k0 / group;
  const uint16_t sc = scales[scale_index(g, n, G_rows)];
  const uint32_t z = zero8_of(zeros, g, n, G_rows);
  const uint32_t s2 = dup16(sc), zm2 = zero_magic2<false>(z);
  const float sf = BF16 ? __uint_as_float(static_cast<uint32_t>(sc) << 16) : __half2float(__ushort_as_half(sc));
  const uint4 v = *reinterpret_cast<const uint4 *>(qw + c * 16);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t d[2];
    dequant_word8<BF16>(w[j], fp8 != 0, zm2, z, s2, sf, d);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const size_t k = static_cast<size_t>(k0 + 4 * j + 2 * i);
      out[k * N + n] = static_cast<uint16_t>(d[i] & 0xFFFFu);
      out[(k + 1) * N + n] = static_cast<uint16_t>(d[i] >> 16);
    }
  }
}

cudaError_t launch_repack8(const uint8_t *q, uint8_t *qw, int K, int N, cudaStream_t st) {
  const size_t total = static_cast<size_t>(K) * N / 16;
  repack8_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(q, qw, K, N);
  return cudaGetLastError();
}

cudaError_t launch_pack_zeros8(const uint8_t *z, uint8_t *zp, int rows, int N, int rep, cudaStream_t st) {
  const size_t total = static_cast<size_t>(rows) * N;
  pack_zeros8_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(z, zp, rows, N, rep);
  return cudaGetLastError();
}

cudaError_t launch_dequant8(const uint8_t *qw, const uint16_t *scales, const uint8_t *zeros, bool fp8,
                            uint16_t *out, int K, int N, int group, bool bf16, cudaStream_t st) {
  const size_t total = static_cast<size_t>(K) * N / 16;
  const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
  if (bf16)
    dequant8_kernel<true><<<blocks, 256, 0, st>>>(qw, scales, zeros, fp8 ? 1 : 0, out, K, N, group);
  else
    dequant8_kernel<false><<<blocks, 256, 0, st>>>(qw, scales, zeros, fp8 ? 1 : 0, out, K, N, group);
  return cudaGetLastError();
}

cudaError_t launch_repack(const void *q, uint8_t *qw, int K, int N, int src, unsigned int *err,
                          cudaStream_t st) {
  dim3 grid(N / ATOM_N, K / ATOM_K);
  const uint8_t *qb = static_cast<const uint8_t *>(q);
  switch (src) {
    case SRC_U8: repack_kernel<SRC_U8><<<grid, 256, 0, st>>>(qb, qw, K, N, err); break;
    case SRC_AWQ: repack_kernel<SRC_AWQ><<<grid, 256, 0, st>>>(qb, qw, K, N, err); break;
    case SRC_GPTQ: repack_kernel<SRC_GPTQ><<<grid, 256, 0, st>>>(qb, qw, K, N, err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_zeros(const void *z, uint8_t *zp, int rows, int N, int rep, int src, int offset,
                              unsigned int *err, cudaStream_t st) {
  const size_t total = static_cast<size_t>(rows) * (N / 2);
  const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
  const uint8_t *zb = static_cast<const uint8_t *>(z);
  switch (src) {
    case SRC_U8: pack_zeros_kernel<SRC_U8><<<blocks, 256, 0, st>>>(zb, zp, rows, N, rep, offset, err); break;
    case SRC_AWQ: pack_zeros_kernel<SRC_AWQ><<<blocks, 256, 0, st>>>(zb, zp, rows, N, rep, offset, err); break;
    case SRC_GPTQ: pack_zeros_kernel<SRC_GPTQ><<<blocks, 256, 0, st>>>(zb, zp, rows, N, rep, offset, err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_scales(const uint16_t *s, uint16_t *sp, int rows, int N, int rep, cudaStream_t st) {
  const size_t total = static_cast<size_t>(rows) * N;
  const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
  pack_scales_kernel<<<blocks, 256, 0, st>>>(s, sp, rows, N, rep);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t *qw, const uint16_t *scales, const uint8_t *zeros,
                           uint16_t *out, int K, int N, int group, bool bf16, cudaStream_t st) {
  const size_t nchunks = static_cast<size_t>(K) * N / 32;
  const unsigned blocks = static_cast<unsigned>((nchunks + 255) / 256);
  if (bf16)
    dequant_kernel<true><<<blocks, 256, 0, st>>>(qw, scales, zeros, out, K, N, group);
  else
    dequant_kernel<false><<<blocks, 256, 0, st>>>(qw, scales, zeros, out, K, N, group);
  return cudaGetLastError();
}

}  // namespace tmw4

// decode_mma.cu -- persistent stream-K kernel for small row counts (M <= 16)
// whose multiply-accumulate runs on the tensor cores with register operands.
//
// At decode sizes the GEMM is bound by HBM: every packed weight byte is
// used M times, and the kernel must keep enough weight bytes in flight while
// spending as few instructions per packed 32-bit word (eight weights) as it
// can.  Per block of 64 K x 128 columns a CTA
//   * streams the packed weights through a per-warp shared-memory ring with
//     16-byte cp.async copies (DM_DEPTH - 1 blocks in flight per warp; the
//     group's scales and zeros travel in the same ring);
//   * turns each thread's codes into (q - z) exactly in 16-bit floats
//     (exponent-magic OR, then one exact subtract; TurboMind paper,
//     pith.science review, Figure 6: integer-to-float conversion before the
//     scaling);
//   * feeds them to mma.sync m16n8k16 as the A operand (16 weight columns x
//     16 K); the activations are the B operand (8 rows per n8 tile), read
//     straight from global memory (L1-cached, one step ahead): with the K
//     order below, a thread's B fragment of one 16-K step is 8 contiguous
//     bytes of one activation row;
//   * accumulates one quantization group in fp32 and scales it once:
//     C += s * sum_k a_k (q_k - z).  With s applied in fp32 the only
//     roundings are those of the fp32 sums and the final one to 16 bits.
// The K order inside each MMA is a permutation of the actual K order that
// both operands share: thread (g, t) of the fragment layout holds, for
// every column it owns, the 16 consecutive K values [16t, 16t + 16) of a
// 64-K block -- exactly half of one 16-byte chunk of the packed layout (a
// chunk is 32 consecutive K of one column) -- and reads the activations
// with the same mapping.  No shuffle is needed on either side.
//
// Work split (stream-K): the units are (128-column tile, quantization
// group) pairs in tile-major order, and a persistent grid of CTAs -- as many
// as are resident on the GPU at once -- takes equal contiguous ranges of
// them.  Because the packed layout is tile-major, a CTA's weights are one
// contiguous byte range.  A CTA's range covers the end of one tile, whole
// tiles and the start of another; a whole tile is written directly, a cut
// one as an fp32 partial per contributor, and after every CTA of the tile
// has published its partial (one acq_rel atomic each, issued when the CTA
// has finished its range so that no warp waits for it mid-stream) the last
// one to arrive adds the partials in contributor order.  Results do not
// depend on scheduling.
//
// CTA: 4 warps; warp w owns columns 32w + 8c + g (c = 0..3) of the current
// tile: m16 tile mt holds columns c = 2mt (rows g) and c = 2mt + 1 (rows
// g + 8).
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tc_epilogue.cuh"
#include "tmw4_device.cuh"

namespace tmw4 {

// Debug builds (-DTMW4_TRACE): %globaltimer of CTA-level events of the first
// 2048 CTAs into GemmArgs::trace[event * 2048 + CTA], the CTA's SM in slot 7.
#ifdef TMW4_TRACE
#define DM_TRACE(ev)                                                                           \
  do {                                                                                         \
    const unsigned cta_ = blockIdx.x + gridDim.x * blockIdx.y;                                 \
    if (p.trace != nullptr && threadIdx.x == 0 && cta_ < 2048) {                               \
      p.trace[(ev) * 2048 + cta_] = static_cast<long long>(globaltimer_ns());                  \
      unsigned smid_;                                                                          \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));                                       \
      p.trace[7 * 2048 + cta_] = smid_;                                                        \
    }                                                                                          \
  } while (0)
#else
#define DM_TRACE(ev) \
  do {               \
  } while (0)
#endif

namespace {

constexpr int DM_CONSUMERS = 128;   // four warps that dequantize and multiply
constexpr int DM_THREADS = 160;     // + one producer warp
constexpr int DM_DEPTH = 8;         // ring stages: up to DM_DEPTH blocks in flight
constexpr int DM_W_BYTES = 4096;    // one 64-K block of the tile's packed weights
constexpr int DM_META_BYTES = 320;  // a group's scales (256 B) and zeros (64 B) for the tile

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

}  // namespace

// Shared memory of a CTA: a ring of DM_DEPTH stages filled by the producer
// warp with TMA copies, one stage per 64-K block:
//   activations   [8 NT8 rows][128 B] (TMA tensor copy, 128-byte swizzle:
//                 16-byte chunk c of row r sits at chunk c ^ (r % 8); rows
//                 past M are filled with zeros by the copy);
//   weights       the block's 4096 packed bytes as stored (one bulk copy);
//   group data    the tile's 128 scales (256 B) and 64 zero bytes, in the
//                 stage of the block that starts a group (two bulk copies).
// full[s] completes when a stage has landed (transaction bytes), empty[s]
// when the four consumer warps have read it.
__host__ __device__ constexpr int dm_stage_bytes(int nt8) {
  return (1024 * nt8 + DM_W_BYTES + DM_META_BYTES + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int dm_smem_bytes(int nt8) { return DM_DEPTH * dm_stage_bytes(nt8) + 1024; }

// NT8: n8 tiles of activation rows (M <= 8 * NT8).  GS: 64-K blocks per
// quantization group (1 for G = 64, 2 for G = 128).
//
// Fragment roles (mma.sync m16n8k16, row.col): A = dequantized weights (16
// columns x 16 K), B = activations (16 K x 8 rows), D = C^T tile in fp32.
// For 16-K step i of a 64-K block, thread (g, t) holds
//   a0, a2 = pairs 2(i%2), 2(i%2)+1 of word i/2 of its slice of column c = 2mt
//   a1, a3 = the same pairs of column c = 2mt + 1
//            (actual K 16t + 4i + {0,1} and 16t + 4i + {2,3})
//   b0, b1 = activation row 8 j8 + g at the same K: 8 contiguous bytes.
// CL selects the work split:
//   false  stream-K over a persistent grid (above): fp32 partials of cut
//          tiles in the workspace, reduced by the last CTA to arrive;
//   true   split-K inside a thread-block cluster: grid (tiles, S) in clusters
//          of (1, S, 1); rank r of a cluster takes the r-th of S equal,
//          group-aligned K ranges of the tile; the partials stay in each
//          CTA's shared memory and rank 0 adds them in rank order through
//          distributed shared memory after a bounded mbarrier handshake (no
//          workspace, no atomics).
template <bool BF16, int NT8, int GS, bool CL>
__global__ void __launch_bounds__(DM_THREADS)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs p) {
  extern __shared__ uint8_t dm_smem_raw[];
  constexpr int D = DM_DEPTH;
  constexpr int STAGE = dm_stage_bytes(NT8);
  constexpr int ACT_BYTES = 1024 * NT8;
  constexpr int W0 = ACT_BYTES, META0 = ACT_BYTES + DM_W_BYTES;
  static_assert((D & (D - 1)) == 0 && STAGE % 1024 == 0, "ring geometry");
  __shared__ uint64_t full_bar[D], empty_bar[D];
  __shared__ uint64_t ready_bar, done_bar;     // cluster mode: partials ready / read
  __shared__ int seg_tile[2], seg_last[2];
  __shared__ int abort_flag_s;
  volatile int *abort_flag = &abort_flag_s;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(dm_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = p.K / 64;
  const int GR = p.K / p.group;                    // groups (units) per tile
  const long long U = static_cast<long long>(p.N / TILE_N) * GR;
  const long long Gc = gridDim.x;
  // this CTA's blocks: nb consecutive 64-K blocks from block b0 (tile-major)
  long long u0, b0;
  int nb;
  uint32_t rank = 0;
  const int S = CL ? static_cast<int>(gridDim.y) : 1;
  if constexpr (CL) {
    rank = cluster_ctarank();
    const int kb_start = static_cast<int>(rank) * p.kb_per_split;
    nb = max(0, min(KB, kb_start + p.kb_per_split) - kb_start);
    b0 = static_cast<long long>(blockIdx.x) * KB + kb_start;
    u0 = b0 / GS;
  } else {
    u0 = unit_begin(blockIdx.x, U, Gc);
    nb = static_cast<int>(unit_begin(blockIdx.x + 1, U, Gc) - u0) * GS;
    b0 = u0 * GS;
  }
  const bool has_zeros = p.zeros != nullptr;
  const int M = p.M, N = p.N;

  if (threadIdx.x < D) {
    mbar_init(full_bar + threadIdx.x, 1);
    mbar_init(empty_bar + threadIdx.x, 4);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) {
    abort_flag_s = 0;
    if constexpr (CL) {
      mbar_init(&ready_bar, static_cast<uint32_t>(S > 1 ? S - 1 : 1));
      mbar_init(&done_bar, 1);
      fence_mbar_init();
    }
  }
  __syncwarp();
  if constexpr (CL) {
    cluster_sync();   // every barrier of the cluster is initialised before any remote arrival
  } else {
    __syncthreads();
  }
  pdl_launch_dependents();
  DM_TRACE(0);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_a);
      const int nfirst = min(nb, D);
      int kb = static_cast<int>(b0 % KB);
      auto copy_weights = [&](int i) {
        uint8_t *st = smem + (i & (D - 1)) * STAGE;
        const bool grp = i % GS == 0;
        mbar_arrive_expect_tx(full_bar + (i & (D - 1)),
                              ACT_BYTES + DM_W_BYTES + (grp ? 256 + (has_zeros ? 64 : 0) : 0));
        tma_bulk_g2s(st + W0, p.qw + (b0 + i) * BLOCK_BYTES, DM_W_BYTES, full_bar + (i & (D - 1)));
        if (grp) {
          const long long u = u0 + i / GS;
          tma_bulk_g2s(st + META0, p.scales + u * TILE_N, 256, full_bar + (i & (D - 1)));
          if (has_zeros) tma_bulk_g2s(st + META0 + 256, p.zeros + u * (TILE_N / 2), 64, full_bar + (i & (D - 1)));
        }
      };
      auto copy_acts = [&](int i, int kbi) {
        uint8_t *st = smem + (i & (D - 1)) * STAGE;
        if (p.act_map_3d)
          tma_load_3d(st, &tmap_a, 0, 0, kbi, full_bar + (i & (D - 1)));
        else
          tma_load_2d(st, &tmap_a, kbi * 64, 0, full_bar + (i & (D - 1)));
      };
      // the packed weights do not depend on earlier kernels in the stream:
      // the first stages' weights are requested before waiting for them,
      // their activations once the previous kernel has completed
      for (int i = 0; i < nfirst; ++i) copy_weights(i);
      pdl_wait();
      for (int i = 0; i < nfirst; ++i) {
        copy_acts(i, kb);
        if (++kb == KB) kb = 0;
      }
      int issued = nfirst;
      for (int i = nfirst; i < nb; ++i) {
        // stage i % D is free once the consumers have read block i - D
        if (!mbar_wait_bounded(empty_bar + (i & (D - 1)), ((i / D) & 1) ^ 1u, p.limit_ns, abort_flag, p.err,
                               SITE_PRODUCER_EMPTY, i))
          break;
        copy_weights(i);
        copy_acts(i, kb);
        if (++kb == KB) kb = 0;
        issued = i + 1;
      }
      // every copy issued must have landed before the CTA exits
      for (int i = max(0, issued - D); i < issued; ++i)
        mbar_wait_bounded(full_bar + (i & (D - 1)), (i / D) & 1, p.limit_ns, nullptr, p.err, SITE_DRAIN_TMA, i);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  float acc[2][NT8][4];
  float accg[2][NT8][4];
  uint32_t zm[4], z16[4];     // per column of the current group: (MAGIC + z), -(64 + z) (fp16)
  float sc[4];                // per column of the current group: the scale
  const int zsh = (g >> 1) * 8 + (g & 1) * 4;
  // this thread's reads in a stage: weights of column 32w + 8c + g at
  // wrd + 128c; scales at mrd + 16c (+ 2 bytes per column), zeros at mzd;
  // B fragment of n8 tile j8, 16-K step i: row 8 j8 + g, chunk (2t + i/2) ^ g
  const int wrd = W0 + (warp >> 1) * ATOM_BYTES + (t >> 1) * 1024 + ((warp & 1) * 32 + g) * 16 + (t & 1) * 8;
  const int mrd = META0 + 2 * (32 * warp + g);
  const int mzd = META0 + 256 + 16 * warp;
  int brd[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) brd[i] = g * 128 + (((2 * t + (i >> 1)) ^ g) << 4) + ((i & 1) << 3);
  int nseg = 0;
  bool ok = true;
  // cut segments of the range (the first and the last may be cut), from the
  // range alone, so that every consumer warp takes the same barriers below
  // even if one of them gave up a wait
  const long long t_first = b0 / KB, t_last = (b0 + nb - 1) / KB;
  const bool first_cut = b0 % KB != 0 || b0 + nb < (t_first + 1) * KB;
  const bool last_cut = t_last != t_first && (b0 + nb) % KB != 0;
  const int nseg_range = (first_cut ? 1 : 0) + (last_cut ? 1 : 0);

#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][j8][e] = 0.f;
  int i = 0;
  int kb_c = static_cast<int>(b0 % KB), t_c = static_cast<int>(b0 / KB);
#pragma unroll 1
  while (i < nb && ok) {
    // a tile segment: blocks [i, i + len) of tile t_c
    const int len = min(nb - i, KB - kb_c);
    const bool whole = kb_c == 0 && len == KB;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][j8][e] = 0.f;
#pragma unroll 1
    for (int ig = i; ig < i + len && ok; ig += GS) {
#pragma unroll
      for (int u = 0; u < GS; ++u) {
        const int ib = ig + u;
        const int sidx = ib & (D - 1);
        if (!mbar_wait_warp(full_bar + sidx, (ib / D) & 1, p.limit_ns, abort_flag, p.err, SITE_DQ_FULL, ib)) {
          ok = false;
          break;
        }
        const uint8_t *st = smem + sidx * STAGE;
        uint2 w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint2 *>(st + wrd + 128 * c);
        if (u == 0) {
          // group start: its scales and zero points
          const uint4 zw = has_zeros ? *reinterpret_cast<const uint4 *>(st + mzd) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            sc[c] = bits16_to_f32<BF16>(*reinterpret_cast<const uint16_t *>(st + mrd + 16 * c));
            const uint32_t zwc = c == 0 ? zw.x : c == 1 ? zw.y : c == 2 ? zw.z : zw.w;
            const uint32_t z = has_zeros ? (zwc >> zsh) & 0xFu : 8u;
            zm[c] = z * 0x00010001u + Magic<BF16>::pair;
            z16[c] = z * 0x00100010u + 0xD400D400u;   // fp16 -(64 + z) in both halves
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
              for (int e = 0; e < 4; ++e) accg[mt][j8][e] = 0.f;
        }
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
          uint2 bf[NT8][2];
#pragma unroll
          for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
            for (int j = 0; j < 2; ++j)
              bf[j8][j] = *reinterpret_cast<const uint2 *>(st + j8 * 1024 + brd[2 * wi + j]);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            uint32_t lo[4], hi[4];
            codes_minus_zero<BF16>(wi == 0 ? w[2 * mt].x : w[2 * mt].y, zm[2 * mt], z16[2 * mt], lo);
            codes_minus_zero<BF16>(wi == 0 ? w[2 * mt + 1].x : w[2 * mt + 1].y, zm[2 * mt + 1],
                                   z16[2 * mt + 1], hi);
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int j8 = 0; j8 < NT8; ++j8)
                mma_16816<BF16>(accg[mt][j8], lo[2 * j], hi[2 * j], lo[2 * j + 1], hi[2 * j + 1],
                                bf[j8][j].x, bf[j8][j].y);
          }
        }
        // the stage has been read: release it to the producer
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar + sidx);
        if (u == GS - 1) {
          // end of a group: C += s * sum over the group
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int j8 = 0; j8 < NT8; ++j8) {
              ffma2(acc[mt][j8][0], acc[mt][j8][1], sc[2 * mt], sc[2 * mt], accg[mt][j8][0], accg[mt][j8][1]);
              ffma2(acc[mt][j8][2], acc[mt][j8][3], sc[2 * mt + 1], sc[2 * mt + 1], accg[mt][j8][2],
                    accg[mt][j8][3]);
            }
        }
      }
    }
    if (!ok) break;
    // the segment ends: a whole tile goes to C, a cut one to its contributor
    // slot (published when the range is done).  Accumulator element e of
    // (mt, j8): column col = 32 w + 8 (2 mt + e / 2) + g of tile t_c,
    // activation row m = 8 j8 + 2t + e % 2
    float *part = nullptr;
    if (CL && !whole) break;   // cluster mode: the one segment's sums stay in registers
    if (!whole) {
      const int jc = static_cast<int>(blockIdx.x) - cta_of_unit(static_cast<long long>(t_c) * GR, U, Gc);
      part = p.ws + (static_cast<size_t>(t_c) * p.ws_slots + jc) * M * TILE_N;
      if (threadIdx.x == 0) seg_tile[nseg] = t_c;
      ++nseg;
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = 8 * j8 + 2 * t + (e & 1);
          const int col = 32 * warp + 8 * (2 * mt + (e >> 1)) + g;
          if (m < M) {
            if (whole)
              p.C[static_cast<size_t>(m) * N + static_cast<size_t>(t_c) * TILE_N + col] =
                  f32_to_bits16<BF16>(acc[mt][j8][e]);
            else
              part[m * TILE_N + col] = acc[mt][j8][e];
          }
        }
    i += len;
    kb_c = 0;
    ++t_c;
  }
  DM_TRACE(3);
  (void)nseg;
  if constexpr (CL) {
    if (S == 1) return;   // the whole tile was written
    // Cluster split-K: every consumer thread leaves its 8 NT8 sums at its own
    // slot of this CTA's (now idle) ring; rank 0 adds the slots of ranks
    // 1..S-1 to its own, in rank order, and writes C.  The handshake: each
    // rank's thread 0 arrives on rank 0's ready barrier (release, cluster
    // scope) once its consumers have stored; rank 0 waits for all S - 1,
    // reads, then arrives on every rank's done barrier, which each rank waits
    // for before exiting (its shared memory must outlive the reads).
    // Every wait is bounded.  A rank whose own pipeline gave up still takes
    // part (C is then undefined, the error word says why), and rank 0 waits
    // for the others several times longer than any of them can be held up by
    // its own bounded waits, so that no arrival reaches an exited CTA.
    constexpr int NV = 2 * NT8 * 4;
    float *slot = reinterpret_cast<float *>(smem) + threadIdx.x * NV;
    if (rank != 0) {
      named_bar_sync(1, DM_CONSUMERS);   // no warp still reads the ring
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
          for (int e = 0; e < 4; ++e) slot[(mt * NT8 + j8) * 4 + e] = acc[mt][j8][e];
      named_bar_sync(1, DM_CONSUMERS);
      if (threadIdx.x == 0) {
        mbar_arrive_remote(mapa_shared(smem_u32(&ready_bar), 0));
        mbar_wait_bounded(&done_bar, 0, 16 * p.limit_ns, nullptr, p.err, SITE_CLUSTER_DONE, rank);
      }
      named_bar_sync(1, DM_CONSUMERS);
      return;
    }
    if (threadIdx.x == 0) {
      if (!mbar_wait_bounded(&ready_bar, 0, 8 * p.limit_ns, nullptr, p.err, SITE_CLUSTER_READY, 0))
        *abort_flag = 1;
      fence_acq_rel_cluster();
    }
    named_bar_sync(1, DM_CONSUMERS);
    if (*abort_flag == 0) {
      fence_acq_rel_cluster();
      const uint32_t my_slot = smem_u32(slot);
      for (int r = 1; r < S; ++r) {
        const uint32_t remote = mapa_shared(my_slot, static_cast<uint32_t>(r));
#pragma unroll
        for (int q = 0; q < NV / 4; ++q) {
          const float4 v = ld_shared_cluster_f4(remote + 16 * q);
          float *a = &acc[0][0][0] + 4 * q;
          a[0] += v.x;
          a[1] += v.y;
          a[2] += v.z;
          a[3] += v.w;
        }
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 8 * j8 + 2 * t + (e & 1);
            const int col = 32 * warp + 8 * (2 * mt + (e >> 1)) + g;
            if (m < M)
              p.C[static_cast<size_t>(m) * N + static_cast<size_t>(blockIdx.x) * TILE_N + col] =
                  f32_to_bits16<BF16>(acc[mt][j8][e]);
          }
    }
    // every rank may leave once rank 0 is done with its shared memory
    named_bar_sync(1, DM_CONSUMERS);
    if (threadIdx.x == 0)
      for (int r = 1; r < S; ++r) mbar_arrive_remote(mapa_shared(smem_u32(&done_bar), static_cast<uint32_t>(r)));
    return;
  }
  if (nseg_range == 0) return;   // every tile the range touches was whole

  // publish the cut segments: the barrier orders every consumer's partial
  // writes before one thread's release-acquire arrival per tile (cumulative
  // release); the second barrier passes the outcome (and the acquire) on.
  // After a wait gave up (the abort flag; C is then undefined and the error
  // is reported by tm_poll_error) nothing is published.
  named_bar_sync(1, DM_CONSUMERS);
  const bool aborted = *abort_flag != 0;
  if (threadIdx.x == 0 && !aborted) {
    // both arrivals are issued before either result is used
    const unsigned prev0 = atomic_add_acq_rel_gpu(p.counters + seg_tile[0], 1u);
    const unsigned prev1 = nseg_range > 1 ? atomic_add_acq_rel_gpu(p.counters + seg_tile[1], 1u) : 0u;
    for (int k = 0; k < nseg_range; ++k) {
      const int tt = seg_tile[k];
      const int ncontrib = cta_of_unit(static_cast<long long>(tt) * GR + GR - 1, U, Gc) -
                           cta_of_unit(static_cast<long long>(tt) * GR, U, Gc) + 1;
      seg_last[k] = (k == 0 ? prev0 : prev1) == static_cast<unsigned>(ncontrib - 1);
    }
  }
  named_bar_sync(1, DM_CONSUMERS);
  DM_TRACE(4);
  if (aborted) return;
  for (int k = 0; k < nseg_range; ++k) {
    if (!seg_last[k]) continue;
    // the last contributor of tile tt adds all partials in contributor order
    const int tt = seg_tile[k];
    const int ncontrib = cta_of_unit(static_cast<long long>(tt) * GR + GR - 1, U, Gc) -
                         cta_of_unit(static_cast<long long>(tt) * GR, U, Gc) + 1;
    // Thread x adds the float4s x + 128 r (r < R) of each partial: 4
    // consecutive columns of one row.  QB contributors' loads are issued
    // before any of them is added, so that a reduction costs about
    // ncontrib / QB L2 round trips; the sums still run in contributor order.
    const float *base = p.ws + static_cast<size_t>(tt) * p.ws_slots * M * TILE_N;
    constexpr int RMAX = 2 * NT8;          // float4s per thread per partial (M <= 8 NT8)
    constexpr int QB = 8 / RMAX;
    const int R = (M * (TILE_N / 4) + DM_CONSUMERS - 1) / DM_CONSUMERS;
    float4 sum[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) sum[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < ncontrib; q0 += QB) {
      float4 v[QB][RMAX];
#pragma unroll
      for (int q = 0; q < QB; ++q)
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          const int f4 = threadIdx.x + DM_CONSUMERS * r;
          v[q][r] = (q0 + q < ncontrib && r < R && f4 < M * (TILE_N / 4))
                        ? __ldcg(reinterpret_cast<const float4 *>(base + static_cast<size_t>(q0 + q) * M * TILE_N) + f4)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int q = 0; q < QB; ++q)
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          sum[r].x += v[q][r].x;
          sum[r].y += v[q][r].y;
          sum[r].z += v[q][r].z;
          sum[r].w += v[q][r].w;
        }
    }
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      const int f4 = threadIdx.x + DM_CONSUMERS * r;
      if (r < R && f4 < M * (TILE_N / 4)) {
        const int m = f4 / (TILE_N / 4), col = 4 * (f4 % (TILE_N / 4));
        const uint32_t lo = f32_to_bits16<BF16>(sum[r].x) | (static_cast<uint32_t>(f32_to_bits16<BF16>(sum[r].y)) << 16);
        const uint32_t hi = f32_to_bits16<BF16>(sum[r].z) | (static_cast<uint32_t>(f32_to_bits16<BF16>(sum[r].w)) << 16);
        *reinterpret_cast<uint2 *>(p.C + static_cast<size_t>(m) * N + static_cast<size_t>(tt) * TILE_N + col) =
            make_uint2(lo, hi);
      }
    }
    if (threadIdx.x == 0) p.counters[tt] = 0u;
  }
  DM_TRACE(5);
}

template <bool BF16, int NT8, int GS>
static cudaError_t launch_dm_t(const GemmArgs &a, const CUtensorMap &tmap, int grid, int cluster,
                               cudaStream_t st) {
  const size_t smem = static_cast<size_t>(dm_smem_bytes(NT8));
  if (cluster > 0) {
    auto kern = decode_mma_kernel<BF16, NT8, GS, true>;
    cudaError_t e = cluster_optin<decode_mma_kernel<BF16, NT8, GS, true>>(dm_smem_bytes(NT8));
    if (e != cudaSuccess) return e;
    return launch_kernel_cluster(kern, dim3(grid, cluster), dim3(DM_THREADS), smem, st, a.pdl != 0,
                                 static_cast<unsigned>(cluster), tmap, a);
  }
  auto kern = decode_mma_kernel<BF16, NT8, GS, false>;
  cudaError_t e = smem_optin<decode_mma_kernel<BF16, NT8, GS, false>>(dm_smem_bytes(NT8));
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(DM_THREADS), smem, st, a.pdl != 0, tmap, a);
}

template <bool BF16, int NT8>
static cudaError_t launch_dm_g(const GemmArgs &a, const CUtensorMap &tmap, int grid, int cluster,
                               cudaStream_t st) {
  return a.group == 64 ? launch_dm_t<BF16, NT8, 1>(a, tmap, grid, cluster, st)
                       : launch_dm_t<BF16, NT8, 2>(a, tmap, grid, cluster, st);
}

// Resident CTAs per SM of the kernel instantiation for (bf16, M, group).
template <bool BF16, int NT8, int GS>
static int dm_occupancy_t() {
  static std::once_flag once[kMaxOptinDevices];
  static int occ[kMaxOptinDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxOptinDevices) return 1;
  std::call_once(once[dev], [&] {
    int v = 0;
    if (smem_optin<decode_mma_kernel<BF16, NT8, GS, false>>(dm_smem_bytes(NT8)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, decode_mma_kernel<BF16, NT8, GS, false>,
                                                      DM_THREADS, dm_smem_bytes(NT8)) != cudaSuccess ||
        v <= 0)
      v = 1;
    occ[dev] = v;
  });
  return occ[dev];
}

template <bool BF16, int NT8>
static int dm_occupancy_g(int group) {
  return group == 64 ? dm_occupancy_t<BF16, NT8, 1>() : dm_occupancy_t<BF16, NT8, 2>();
}

int decode_mma_nt8(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : 0; }

int decode_mma_ctas_per_sm(bool bf16, int M, int group) {
  switch (decode_mma_nt8(M)) {
    case 1: return bf16 ? dm_occupancy_g<true, 1>(group) : dm_occupancy_g<false, 1>(group);
    case 2: return bf16 ? dm_occupancy_g<true, 2>(group) : dm_occupancy_g<false, 2>(group);
    default: return 1;
  }
}

void decode_mma_plan(int M, int N, int K, int group, int max_ctas, int *grid, long long *tiles,
                     int *slots) {
  const long long GR = K / group;
  const long long T = N / TILE_N;
  const long long U = T * GR;
  const long long G = std::max<long long>(1, std::min<long long>(max_ctas, U));
  int maxc = 1;
  for (long long t = 0; t < T; ++t) {
    const int c = cta_of_unit((t + 1) * GR - 1, U, G) - cta_of_unit(t * GR, U, G) + 1;
    if (c > maxc) maxc = c;
  }
  *grid = static_cast<int>(G);
  *tiles = T;
  *slots = maxc;
  (void)M;
}

// Whether clusters of S CTAs (1..16) of the cluster-mode instantiation can
// be resident at all; computed once per (device, S).
template <bool BF16, int NT8, int GS>
static bool dm_cluster_fits_t(int S) {
  static std::once_flag once[kMaxOptinDevices][17];
  static bool fits[kMaxOptinDevices][17];
  int dev = 0;
  if (S < 1 || S > 16 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxOptinDevices) return false;
  std::call_once(once[dev][S], [&] {
    fits[dev][S] = false;
    if (cluster_optin<decode_mma_kernel<BF16, NT8, GS, true>>(dm_smem_bytes(NT8)) != cudaSuccess) return;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, S);
    cfg.blockDim = dim3(DM_THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(dm_smem_bytes(NT8));
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 1;
    attr.val.clusterDim.y = S;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    fits[dev][S] = cudaOccupancyMaxActiveClusters(&n, decode_mma_kernel<BF16, NT8, GS, true>, &cfg) ==
                       cudaSuccess &&
                   n > 0;
    (void)cudaGetLastError();
  });
  return fits[dev][S];
}

template <bool BF16, int NT8>
static bool dm_cluster_fits_g(int group, int S) {
  return group == 64 ? dm_cluster_fits_t<BF16, NT8, 1>(S) : dm_cluster_fits_t<BF16, NT8, 2>(S);
}

int decode_mma_cluster_split(bool bf16, int M, int K, int group, int requested, int *kb_per_split) {
  const int KB = K / 64, GS = group / 64;
  const int req = std::max(1, std::min(requested, 16));
  int per = (KB + req - 1) / req;
  per = (per + GS - 1) / GS * GS;
  const int S = (KB + per - 1) / per;
  bool fits = false;
  switch (decode_mma_nt8(M)) {
    case 1: fits = bf16 ? dm_cluster_fits_g<true, 1>(group, S) : dm_cluster_fits_g<false, 1>(group, S); break;
    case 2: fits = bf16 ? dm_cluster_fits_g<true, 2>(group, S) : dm_cluster_fits_g<false, 2>(group, S); break;
    default: break;
  }
  if (!fits) return 0;
  *kb_per_split = per;
  return S;
}

cudaError_t launch_decode_mma(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int grid,
                              int cluster, cudaStream_t st) {
  switch (decode_mma_nt8(a.M)) {
    case 1:
      return bf16 ? launch_dm_g<true, 1>(a, tmap_a, grid, cluster, st)
                  : launch_dm_g<false, 1>(a, tmap_a, grid, cluster, st);
    case 2:
      return bf16 ? launch_dm_g<true, 2>(a, tmap_a, grid, cluster, st)
                  : launch_dm_g<false, 2>(a, tmap_a, grid, cluster, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tmw4

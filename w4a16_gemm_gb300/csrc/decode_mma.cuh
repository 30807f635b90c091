// decode_mma.cuh -- kernel for small row counts (M <= 16) whose
// multiply-accumulate runs on the tensor cores with register operands, for
// 4-bit or 8-bit codes (template WB).  decode_mma.cu instantiates the
// 4-bit kernels and holds the entry points; decode_mma8.cu instantiates the
// 8-bit ones (two translation units compile in parallel).
//
// At decode sizes the GEMM is bound by HBM: every packed weight byte is
// used M times, and the kernel must keep enough weight bytes in flight while
// spending as few instructions per packed 32-bit word (eight weights) as it
// can.  Per block of 64 K x 128 columns a CTA
//   * has a producer warp stream the packed weights, the group's scales and
//     zeros (bulk copies) and the activation block (a TMA tensor copy) into a
//     shared-memory ring;
//   * turns each consumer thread's codes into (q - z) exactly in 16-bit
//     floats (exponent-magic OR, then one exact subtract; TurboMind paper,
//     pith.science review, Figure 6: integer-to-float conversion before the
//     scaling);
//   * feeds them to mma.sync m16n8k16 as the A operand (16 weight columns x
//     16 K); the activations are the B operand (8 rows per n8 tile);
//   * accumulates one quantization group in fp32 and scales it once:
//     C += s * sum_k a_k (q_k - z).  With s applied in fp32 the only
//     roundings are those of the fp32 sums and the final one to 16 bits.
// The K order inside each MMA is a permutation of the actual K order that
// both operands share: the weights are read with ldmatrix, whose eight row
// addresses are eight consecutive 16-byte chunks (eight columns), so that
// thread (g, t) receives word t of a chunk of column g -- 8 consecutive K
// of a 32-K chunk (4-bit) or 4 consecutive K of a 16-K chunk (8-bit) -- and
// the activations are read with the same mapping.  No shuffle is needed on
// either side, and the shared-memory reads hit distinct banks.
//
// Work split (stream-K): the units are (128-column tile, quantization
// group) pairs in tile-major order, and a persistent grid of CTAs -- as many
// as are resident on the GPU at once, or fewer -- takes equal contiguous
// ranges of them.  Because the packed layout is tile-major, a CTA's weights
// are one contiguous byte range.  A CTA's range covers the end of one tile,
// whole tiles and the start of another; a whole tile is written directly, a
// cut one as an fp32 partial per contributor, and after every CTA of the
// tile has published its partial (one acq_rel atomic each, issued when the
// CTA has finished its range so that no warp waits for it mid-stream) the
// last one to arrive adds the partials in a fixed order.  Results do not
// depend on scheduling.  A second split, thread-block clusters with a
// distributed-shared-memory reduction, is described at the kernel.
//
// Consumer warps come in K-groups of four; warp w of a K-group owns columns
// 32w + 8c + g (c = 0..3) of the current tile: m16 tile mt holds columns
// c = 2mt (rows g) and c = 2mt + 1 (rows g + 8).
#pragma once

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "mma_frag.cuh"
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
// The same from whichever thread calls it.
#define DM_TRACE_ANY(ev)                                                                       \
  do {                                                                                         \
    const unsigned cta_ = blockIdx.x + gridDim.x * blockIdx.y;                                 \
    if (p.trace != nullptr && cta_ < 2048) p.trace[(ev) * 2048 + cta_] = static_cast<long long>(globaltimer_ns()); \
  } while (0)
#else
#define DM_TRACE(ev) \
  do {               \
  } while (0)
#define DM_TRACE_ANY(ev) \
  do {                   \
  } while (0)
#endif

namespace {

// Bytes of one 64-K block of a tile's packed weights (WB bits per code) and
// of a group's zero points for the tile (nibbles for 4 bits, bytes for 8).
template <int WB>
struct DmBytes {
  static constexpr int W = 4096 * WB / 4;
  static constexpr int Z = WB == 8 ? 128 : 64;
  static constexpr int META = 256 + Z;   // + the group's 128 16-bit scales
};

}  // namespace

// Shared memory of a CTA: a ring of D stages, one 64-K block each, filled
// by the producer warp with TMA copies, then a scratch area:
//   [0, D ACT)          activations of stage s at s ACT, ACT = 1024 NT8 bytes:
//                       [8 NT8 rows][128 B] by a TMA tensor copy with the
//                       128-byte swizzle (16-byte chunk c of row r sits at
//                       chunk c ^ (r % 8)); rows past M are zero-filled
//   [W_OFF, + D WM)     the block's 4096 packed weight bytes as stored (one
//                       bulk copy) and, in the stage of a group's first block,
//                       the tile's 128 scales (256 B) and 64 zero bytes
//   [RED_OFF, + RED)    sums of K-groups 1..KG-1 at a segment's end; group
//                       sums of the split-K reduction
//   [RECV_OFF, ...)     cluster mode, rank 0: the other ranks' sums
// full[s] completes when a stage has landed (transaction bytes), empty[s]
// when the four consumer warps that read it are done.  D grows with the
// number of K-groups so that a CTA keeps about as many bytes in flight as
// the SM's share of HBM bandwidth times the load latency asks for.
template <int NT8, int KG, bool CL = false, int WB = 4>
struct DmGeom {
  // (a cluster CTA takes a short K range: a shallower ring leaves room for
  // the receive area and more CTAs per SM; 8-bit stages are twice as large,
  // so half as many keep the same bytes in flight)
  static constexpr int D4 = (KG == 1 || CL) ? 8 : KG == 2 ? 16 : (NT8 == 1 ? 32 : 28);
  static constexpr int D = WB == 8 ? D4 / 2 : D4;
  static constexpr int ACT = 1024 * NT8;
  static constexpr int WM = DmBytes<WB>::W + DmBytes<WB>::META;
  static constexpr int NV = 8 * NT8;            // accumulator floats per consumer thread
  static constexpr int CONS = 128 * KG;         // consumer threads
  static constexpr int RED_KG = (KG - 1) * 128 * NV * 4;
  static constexpr int RED_SK = CONS * 16;
  static constexpr int RED = RED_KG > RED_SK ? RED_KG : RED_SK;
  static constexpr int W_OFF = D * ACT;
  static constexpr int RED_OFF = (W_OFF + D * WM + 127) / 128 * 128;
  static constexpr int RECV_OFF = RED_OFF + RED;
  static constexpr int SMEM = RECV_OFF + 1024;   // + slack to align the base to 1024
};

// Cluster mode: rank 0 receives the other ranks' sums of the rows < M,
// [S - 1][M][128] fp32, behind the scratch area; at most this many bytes.
constexpr int DM_RECV_MAX = 48 * 1024;
__host__ __device__ constexpr int dm_recv_bytes(int M, int S) { return (S - 1) * M * TILE_N * 4; }

// NT8: n8 tiles of activation rows (M <= 8 NT8).  GS: 64-K blocks per
// quantization group (1 for G = 64, 2 for G = 128).  KG: K-groups of four
// consumer warps; K-group j takes the j-th of every KG consecutive groups of
// the CTA's range, and the K-groups add their sums through shared memory at
// the end of each tile segment (in K-group order), so that a tile needs KG
// times fewer CTAs for the same number of warps in flight.
//
// Fragment roles (mma.sync m16n8k16, row.col): A = dequantized weights (16
// columns x 16 K), B = activations (16 K x 8 rows), D = C^T tile in fp32.
// For 16-K step i of a 64-K block, thread (g, t) holds
//   a0, a2 = pairs 2(i%2), 2(i%2)+1 of word t of 32-K chunk i/2 of column c = 2mt
//   a1, a3 = the same pairs of column c = 2mt + 1
//            (actual K 32(i/2) + 8t + 4(i%2) + {0,1} and ... + {2,3})
//   b0, b1 = activation row 8 j8 + g at the same K: 8 contiguous bytes.
// With 8-bit codes (WB = 8) the order differs: step i takes the 16-byte
// chunk i of each column (K 16i..16i+15, loaded with ldmatrix), thread t its
// bytes 4t..4t+3 (actual K 16i + 4t + {0,1} and 16i + 4t + {2,3}).
// CL selects the work split:
//   false  stream-K over a persistent grid (above): fp32 partials of cut
//          tiles in the workspace, reduced by the last CTA to arrive;
//   true   split-K inside a thread-block cluster: grid (tiles, S) in clusters
//          of (1, S, 1); rank r of a cluster takes the r-th of S equal,
//          group-aligned K ranges of the tile; ranks 1..S-1 store their sums
//          of the rows < M into rank 0's shared memory (distributed shared
//          memory), and after one cluster barrier rank 0 adds them in rank
//          order (no workspace, no atomics).  One or two K-groups.
template <bool BF16, int NT8, int GS, bool CL, int KG, int WB>
__global__ void __launch_bounds__(128 * KG + 32, KG == 1 ? (WB == 8 ? 3 : 4) : KG == 2 ? (WB == 8 ? 1 : 2) : 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs p) {
  using Geo = DmGeom<NT8, KG, CL, WB>;
  constexpr int W_BYTES = DmBytes<WB>::W, Z_BYTES = DmBytes<WB>::Z;
  constexpr int D = Geo::D, ACT = Geo::ACT, WM = Geo::WM, NV = Geo::NV, CONS = Geo::CONS;
  static_assert(!CL || KG <= 2, "cluster mode has one or two K-groups");
  static_assert(D <= CONS, "barrier initialisation");
  extern __shared__ uint8_t dm_smem_raw[];
  __shared__ uint64_t full_bar[D], empty_bar[D];
  __shared__ int seg_tile[2], seg_last[2];
  __shared__ int abort_flag_s;
  volatile int *abort_flag = &abort_flag_s;
  uint8_t *smem = align_smem_1024(dm_smem_raw);
  uint8_t *const wm_ring = smem + Geo::W_OFF;
  float *const red = reinterpret_cast<float *>(smem + Geo::RED_OFF);

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
  if (threadIdx.x == 0) abort_flag_s = 0;
  __syncwarp();
  if constexpr (CL) {
    cluster_sync();   // every CTA of the cluster runs before any remote store
  } else {
    __syncthreads();
  }
  pdl_launch_dependents();
  DM_TRACE(0);

  if (warp == 4 * KG) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_a);
      const int nfirst = min(nb, D);
      int kb = static_cast<int>(b0 % KB);
      auto copy_weights = [&](int i) {
        const int s = i % D;
        uint8_t *wm = wm_ring + s * WM;
        const bool grp = i % GS == 0;
        mbar_arrive_expect_tx(full_bar + s, ACT + W_BYTES + (grp ? 256 + (has_zeros ? Z_BYTES : 0) : 0));
        tma_bulk_g2s(wm, p.qw + (b0 + i) * W_BYTES, W_BYTES, full_bar + s);
        if (grp) {
          const long long u = u0 + i / GS;
          tma_bulk_g2s(wm + W_BYTES, p.scales + u * TILE_N, 256, full_bar + s);
          if (has_zeros) tma_bulk_g2s(wm + W_BYTES + 256, p.zeros + u * Z_BYTES, Z_BYTES, full_bar + s);
        }
      };
      auto copy_acts = [&](int i, int kbi) {
        const int s = i % D;
        if (p.act_map_3d)
          tma_load_3d(smem + s * ACT, &tmap_a, 0, 0, kbi, full_bar + s);
        else
          tma_load_2d(smem + s * ACT, &tmap_a, kbi * 64, 0, full_bar + s);
      };
      // the packed weights do not depend on earlier kernels in the stream:
      // the first stages' weights are requested before waiting for them,
      // their activations once the previous kernel has completed
      for (int i = 0; i < nfirst; ++i) copy_weights(i);
      pdl_wait();
      DM_TRACE_ANY(1);
      for (int i = 0; i < nfirst; ++i) {
        copy_acts(i, kb);
        if (++kb == KB) kb = 0;
      }
      int issued = nfirst;
      for (int i = nfirst; i < nb; ++i) {
        // stage i % D is free once the consumers have read block i - D
        if (!mbar_wait_idle(empty_bar + i % D, ((i / D) & 1) ^ 1u, p.limit_ns, abort_flag, p.err,
                            SITE_PRODUCER_EMPTY, i))
          break;
        copy_weights(i);
        copy_acts(i, kb);
        if (++kb == KB) kb = 0;
        issued = i + 1;
      }
      // every copy issued must have landed before the CTA exits
      for (int i = max(0, issued - D); i < issued; ++i)
        mbar_wait_bounded(full_bar + i % D, (i / D) & 1, p.limit_ns, nullptr, p.err, SITE_DRAIN_TMA, i);
    }
    if constexpr (CL) {
      __syncwarp();
      if (S > 1) cluster_sync();   // every thread of the cluster takes the final barrier
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int kg = warp >> 2, wq = warp & 3;          // K-group, column quarter
  const int qtid = threadIdx.x & 127;               // thread within the K-group
  float acc[2][NT8][4];
  float accg[2][NT8][4];
  uint32_t zm[4], z16[4];     // per column of the current group: (MAGIC + z), -(64 + z) (fp16)
  float sc[4];                // per column of the current group: the scale
  float zf[4];                // 8-bit, bf16: 2^23 + z
  const int zsh = (g >> 1) * 8 + (g & 1) * 4;
  // this thread's reads in a stage: weights of column 32 wq + 8c + g at
  // wrd + 128c; scales at mrd + 16c (+ 2 bytes per column), zeros at mzd;
  // B fragment of n8 tile j8, 16-K step i: row 8 j8 + g, chunk (2t + i/2) ^ g
  const int mrd = W_BYTES + 2 * (32 * wq + g);
  const int mzd = WB == 8 ? W_BYTES + 256 + 32 * wq + g : W_BYTES + 256 + 16 * wq;
  int brd[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    brd[i] = WB == 8 ? g * 128 + (((2 * i + (t >> 1)) ^ g) << 4) + ((t & 1) << 3)         // K 16i + 4t + 0..3
                     : g * 128 + (((4 * (i >> 1) + t) ^ g) << 4) + ((i & 1) << 3);        // K 32(i/2) + 8t + 4(i%2) + 0..3
  // ldmatrix row addresses.  8-bit: lane 8m + r gives chunk m of column
  // 32 wq + 8c + r.  4-bit: lane 8mi + r gives chunk (32-K half) mi % 2 of
  // column 32 wq + 8(c0 + mi / 2) + r, for the column pairs c0 = 0 and 2.
  const int ldo = WB == 8 ? 16 * ((lane >> 3) * TILE_N + 32 * wq + (lane & 7))
                          : (wq >> 1) * ATOM_BYTES + ((lane >> 3) & 1) * 1024 +
                                16 * (32 * (wq & 1) + 8 * (lane >> 4) + (lane & 7));
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
  // Every consumer warp walks the same tile segments and takes the same
  // barriers; after a wait gave up (ok = false) it only skips the work.
#pragma unroll 1
  while (i < nb) {
    // a tile segment: blocks [i, i + len) of tile t_c
    const int len = min(nb - i, KB - kb_c);
    const bool whole = kb_c == 0 && len == KB;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][j8][e] = 0.f;
    // this K-group's groups of the segment: range-relative group index = kg (mod KG)
    const int first_ig = i + ((kg - (i / GS) % KG + KG) % KG) * GS;
#pragma unroll 1
    for (int ig = first_ig; ig < i + len && ok; ig += KG * GS) {
#pragma unroll
      for (int u = 0; u < GS; ++u) {
        const int ib = ig + u;
        const int sidx = ib % D;
        if (!mbar_wait_all_idle(full_bar + sidx, (ib / D) & 1, p.limit_ns, abort_flag, p.err, SITE_DQ_FULL, ib)) {
          ok = false;
          break;
        }
#ifdef TMW4_TRACE
        if (ib == 0) DM_TRACE(2);
#endif
        const uint8_t *ast = smem + sidx * ACT;
        const uint8_t *wst = wm_ring + sidx * WM;
        if constexpr (WB == 4) {
          // two ldmatrix: w[c][m] = word t of chunk m (K 32m + 8t + 0..7) of
          // column 32 wq + 8c + g; the eight rows of each matrix are consecutive
          // 16-byte chunks, so the reads hit distinct banks
          uint32_t w[4][2], la[4], lb[4];
          ldmatrix_x4(la, smem_u32(wst) + ldo);
          ldmatrix_x4(lb, smem_u32(wst) + ldo + 256);
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              w[c][m] = la[2 * c + m];
              w[c + 2][m] = lb[2 * c + m];
            }
          if (u == 0) {
            // group start: its scales and zero points
            const uint4 zw = has_zeros ? *reinterpret_cast<const uint4 *>(wst + mzd) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              sc[c] = bits16_to_f32<BF16>(*reinterpret_cast<const uint16_t *>(wst + mrd + 16 * c));
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
                bf[j8][j] = *reinterpret_cast<const uint2 *>(ast + j8 * 1024 + brd[2 * wi + j]);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              uint32_t lo[4], hi[4];
              codes_minus_zero<BF16>(w[2 * mt][wi], zm[2 * mt], z16[2 * mt], lo);
              codes_minus_zero<BF16>(w[2 * mt + 1][wi], zm[2 * mt + 1], z16[2 * mt + 1], hi);
#pragma unroll
              for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int j8 = 0; j8 < NT8; ++j8)
                  mma_16816<BF16>(accg[mt][j8], lo[2 * j], hi[2 * j], lo[2 * j + 1], hi[2 * j + 1],
                                  bf[j8][j].x, bf[j8][j].y);
            }
          }
        } else {
          // 8-bit codes: column c's chunk t holds K 16t..16t+15, word i of it
          // the K of 16-K step i
          // one ldmatrix per column octet c: w8[c][i] = bytes 4t..4t+3 of chunk i
          // (K 16i + 4t + 0..3) of column 32 wq + 8c + g; the eight rows of each
          // matrix are consecutive 16-byte chunks, so the reads hit distinct banks
          uint32_t w8[4][4];
#pragma unroll
          for (int c = 0; c < 4; ++c) ldmatrix_x4(w8[c], smem_u32(wst) + ldo + 128 * c);
          if (u == 0) {
            // group start: its scales and zero points (symmetric int8: 128)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              sc[c] = bits16_to_f32<BF16>(*reinterpret_cast<const uint16_t *>(wst + mrd + 16 * c));
              const uint32_t z = has_zeros ? static_cast<uint32_t>(wst[mzd + 8 * c]) : 128u;
              zm[c] = (0x6400u + z) * 0x00010001u;   // fp16 1024 + z in both halves
              zf[c] = __uint_as_float(0x4B000000u | z);
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
                for (int e = 0; e < 4; ++e) accg[mt][j8][e] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint2 bf[NT8];
#pragma unroll
            for (int j8 = 0; j8 < NT8; ++j8) bf[j8] = *reinterpret_cast<const uint2 *>(ast + j8 * 1024 + brd[i]);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              uint32_t a0, a1, a2, a3;
              codes8_minus_zero<BF16>(w8[2 * mt][i], zm[2 * mt], zf[2 * mt], p.fp8 != 0, a0, a2);
              codes8_minus_zero<BF16>(w8[2 * mt + 1][i], zm[2 * mt + 1], zf[2 * mt + 1], p.fp8 != 0, a1, a3);
#pragma unroll
              for (int j8 = 0; j8 < NT8; ++j8) mma_16816<BF16>(accg[mt][j8], a0, a1, a2, a3, bf[j8].x, bf[j8].y);
            }
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
    if constexpr (KG > 1) {
      // K-groups 1..KG-1 leave their sums in the scratch, K-group 0 adds
      // them in K-group order
      if (kg != 0) {
        float4 *dst = reinterpret_cast<float4 *>(red + ((kg - 1) * 128 + qtid) * NV);
#pragma unroll
        for (int q = 0; q < NV / 4; ++q) dst[q] = *reinterpret_cast<const float4 *>(&acc[0][0][0] + 4 * q);
      }
      named_bar_sync(1, CONS);
      if (kg == 0) {
#pragma unroll 1
        for (int k = 1; k < KG; ++k) {
          const float4 *src = reinterpret_cast<const float4 *>(red + ((k - 1) * 128 + qtid) * NV);
#pragma unroll
          for (int q = 0; q < NV / 4; ++q) {
            const float4 v = src[q];
            float *a = &acc[0][0][0] + 4 * q;
            a[0] += v.x;
            a[1] += v.y;
            a[2] += v.z;
            a[3] += v.w;
          }
        }
      }
    }
    if constexpr (CL) {
      if (!whole) break;   // cluster mode: the one cut segment's sums stay in K-group 0's registers
    }
    // the segment ends: a whole tile goes to C, a cut one to its contributor
    // slot (published when the range is done).  Accumulator element e of
    // (mt, j8): column col = 32 wq + 8 (2 mt + e / 2) + g of tile t_c,
    // activation row m = 8 j8 + 2t + e % 2
    float *part = nullptr;
    if (!whole) {
      const int jc = static_cast<int>(blockIdx.x) - cta_of_unit(static_cast<long long>(t_c) * GR, U, Gc);
      part = p.ws + (static_cast<size_t>(t_c) * p.ws_slots + jc) * M * TILE_N;
      if (threadIdx.x == 0) seg_tile[nseg] = t_c;
      ++nseg;
    }
    if (kg == 0) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 8 * j8 + 2 * t + (e & 1);
            const int col = 32 * wq + 8 * (2 * mt + (e >> 1)) + g;
            if (m < M) {
              if (whole)
                p.C[static_cast<size_t>(m) * N + static_cast<size_t>(t_c) * TILE_N + col] =
                    f32_to_bits16<BF16>(acc[mt][j8][e]);
              else
                part[m * TILE_N + col] = acc[mt][j8][e];
            }
          }
    }
    if constexpr (KG > 1) named_bar_sync(1, CONS);   // the scratch is read before it is written again
    i += len;
    kb_c = 0;
    ++t_c;
  }
  DM_TRACE(3);
  (void)nseg;
  if constexpr (CL) {
    if (S == 1) return;   // the whole tile was written
    // Ranks 1..S-1 store their sums of the rows < M into rank 0's receive
    // area (remote shared-memory stores, which need no reply); the cluster
    // barrier (release / acquire at cluster scope, taken by every thread of
    // every CTA of the cluster, the producer warps included) makes them
    // visible to rank 0, which adds them to its own sums in rank order and
    // writes C.  Rank 0's shared memory outlives every store into it, and no
    // CTA reads another's afterwards, so the other ranks may exit at once.
    // After a wait gave up, the stores and barrier still happen (C is then
    // undefined; the error word says why).
    float *recv = reinterpret_cast<float *>(smem + Geo::RECV_OFF);
    if (rank != 0 && kg == 0) {
      const uint32_t dst = mapa_shared(smem_u32(recv), 0) + (rank - 1) * M * TILE_N * 4;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 8 * j8 + 2 * t + (e & 1);
            const int col = 32 * wq + 8 * (2 * mt + (e >> 1)) + g;
            if (m < M) st_shared_cluster_f32(dst + (m * TILE_N + col) * 4, acc[mt][j8][e]);
          }
    }
    cluster_sync();
    DM_TRACE(4);
    if (rank == 0 && kg == 0 && *abort_flag == 0) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 8 * j8 + 2 * t + (e & 1);
            const int col = 32 * wq + 8 * (2 * mt + (e >> 1)) + g;
            if (m < M) {
              float v = acc[mt][j8][e];
              for (int r = 1; r < S; ++r) v += recv[((r - 1) * M + m) * TILE_N + col];
              p.C[static_cast<size_t>(m) * N + static_cast<size_t>(blockIdx.x) * TILE_N + col] = f32_to_bits16<BF16>(v);
            }
          }
    }
    DM_TRACE(5);
    return;
  }
  if (nseg_range == 0) return;   // every tile the range touches was whole

  // publish the cut segments: the barrier orders every consumer's partial
  // writes before one thread's release-acquire arrival per tile (cumulative
  // release); the second barrier passes the outcome (and the acquire) on.
  // After a wait gave up (the abort flag; C is then undefined and the error
  // is reported by tm_poll_error) nothing is published.
  named_bar_sync(1, CONS);
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
  named_bar_sync(1, CONS);
  DM_TRACE(4);
  if (aborted) return;
  for (int k = 0; k < nseg_range; ++k) {
    if (!seg_last[k]) continue;
    // The last contributor of tile tt adds the partials.  E float4s (4
    // consecutive columns of one row) per partial; P thread groups each add
    // the contributors q = p (mod P) in increasing order, QB contributors'
    // loads in flight at once (a reduction costs about ncontrib / (P QB) L2
    // round trips); the P group sums are then added in group order through
    // shared memory.  The order depends only on the shape: results are
    // reproducible bit for bit.
    const int tt = seg_tile[k];
    const int ncontrib = cta_of_unit(static_cast<long long>(tt) * GR + GR - 1, U, Gc) -
                         cta_of_unit(static_cast<long long>(tt) * GR, U, Gc) + 1;
    const float *base = p.ws + static_cast<size_t>(tt) * p.ws_slots * M * TILE_N;
    const int E = M * (TILE_N / 4);
    int P = 1;
    while (2 * P * E <= CONS && 2 * P <= ncontrib) P *= 2;
    const int TPG = CONS / P;                      // threads per group
    const int pg = threadIdx.x / TPG, el = threadIdx.x % TPG;
    constexpr int RMAX = 2 * NT8 / KG > 0 ? 2 * NT8 / KG : 1;   // float4s per thread per partial
    constexpr int QB = 8 / RMAX;
    float4 sum[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) sum[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = pg; q0 < ncontrib; q0 += P * QB) {
      float4 v[QB][RMAX];
#pragma unroll
      for (int q = 0; q < QB; ++q)
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          const int qq = q0 + q * P, f4 = el + TPG * r;
          v[q][r] = (qq < ncontrib && f4 < E)
                        ? __ldcg(reinterpret_cast<const float4 *>(base + static_cast<size_t>(qq) * M * TILE_N) + f4)
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
    auto store_c = [&](int f4, float4 v) {
      const int m = f4 / (TILE_N / 4), col = 4 * (f4 % (TILE_N / 4));
      const uint32_t lo = f32_to_bits16<BF16>(v.x) | (static_cast<uint32_t>(f32_to_bits16<BF16>(v.y)) << 16);
      const uint32_t hi = f32_to_bits16<BF16>(v.z) | (static_cast<uint32_t>(f32_to_bits16<BF16>(v.w)) << 16);
      *reinterpret_cast<uint2 *>(p.C + static_cast<size_t>(m) * N + static_cast<size_t>(tt) * TILE_N + col) =
          make_uint2(lo, hi);
    };
    if (P == 1) {
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
        if (el + TPG * r < E) store_c(el + TPG * r, sum[r]);
    } else {
      float4 *gs = reinterpret_cast<float4 *>(red);   // [P][E]; P E <= CONS, so one float4 per thread
      if (el < E) gs[pg * E + el] = sum[0];
      named_bar_sync(1, CONS);
      for (int f4 = threadIdx.x; f4 < E; f4 += CONS) {
        float4 v = gs[f4];
        for (int pp = 1; pp < P; ++pp) {
          const float4 w4 = gs[pp * E + f4];
          v.x += w4.x;
          v.y += w4.y;
          v.z += w4.z;
          v.w += w4.w;
        }
        store_c(f4, v);
      }
      named_bar_sync(1, CONS);   // the scratch is read before the next tile's reduction
    }
    if (threadIdx.x == 0) p.counters[tt] = 0u;
  }
  DM_TRACE(5);
}

template <bool BF16, int NT8, int GS, int KG, int WB>
static cudaError_t launch_dm_t(const GemmArgs &a, const CUtensorMap &tmap, int grid, int cluster,
                               cudaStream_t st) {
  constexpr int SMEM = DmGeom<NT8, KG, false, WB>::SMEM;
  const dim3 block(128 * KG + 32);
  if (cluster > 0) {
    if constexpr (KG <= 2) {
      constexpr int CSMEM = DmGeom<NT8, KG, true, WB>::SMEM;
      auto kern = decode_mma_kernel<BF16, NT8, GS, true, KG, WB>;
      cudaError_t e = cluster_optin<decode_mma_kernel<BF16, NT8, GS, true, KG, WB>>(CSMEM + DM_RECV_MAX);
      if (e != cudaSuccess) return e;
      const int recv = dm_recv_bytes(a.M, cluster);
      if (recv > DM_RECV_MAX) return cudaErrorInvalidValue;
      return launch_kernel_cluster(kern, dim3(grid, cluster), block, static_cast<size_t>(CSMEM + recv), st,
                                   a.pdl != 0, static_cast<unsigned>(cluster), tmap, a);
    } else {
      return cudaErrorInvalidValue;
    }
  }
  auto kern = decode_mma_kernel<BF16, NT8, GS, false, KG, WB>;
  cudaError_t e = smem_optin<decode_mma_kernel<BF16, NT8, GS, false, KG, WB>>(SMEM);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), block, static_cast<size_t>(SMEM), st, a.pdl != 0, tmap, a);
}

template <bool BF16, int NT8, int KG, int WB>
static cudaError_t launch_dm_g(const GemmArgs &a, const CUtensorMap &tmap, int grid, int cluster,
                               cudaStream_t st) {
  return a.group == 64 ? launch_dm_t<BF16, NT8, 1, KG, WB>(a, tmap, grid, cluster, st)
                       : launch_dm_t<BF16, NT8, 2, KG, WB>(a, tmap, grid, cluster, st);
}

template <bool BF16, int NT8, int WB>
static cudaError_t launch_dm_k(const GemmArgs &a, const CUtensorMap &tmap, int kgroups, int grid, int cluster,
                               cudaStream_t st) {
  switch (kgroups) {
    case 1: return launch_dm_g<BF16, NT8, 1, WB>(a, tmap, grid, cluster, st);
    case 2: return launch_dm_g<BF16, NT8, 2, WB>(a, tmap, grid, cluster, st);
    case 4:
      if constexpr (WB == 4) return launch_dm_g<BF16, NT8, 4, WB>(a, tmap, grid, cluster, st);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

// Resident CTAs per SM of the stream-K instantiation for (bf16, M, group, KG).
template <bool BF16, int NT8, int GS, int KG, int WB>
static int dm_occupancy_t() {
  static std::once_flag once[kMaxOptinDevices];
  static int occ[kMaxOptinDevices];
  constexpr int SMEM = DmGeom<NT8, KG, false, WB>::SMEM;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxOptinDevices) return 1;
  std::call_once(once[dev], [&] {
    int v = 0;
    if (smem_optin<decode_mma_kernel<BF16, NT8, GS, false, KG, WB>>(SMEM) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, decode_mma_kernel<BF16, NT8, GS, false, KG, WB>,
                                                      128 * KG + 32, SMEM) != cudaSuccess ||
        v <= 0)
      v = 1;
    occ[dev] = v;
  });
  return occ[dev];
}

template <bool BF16, int NT8, int KG, int WB>
static int dm_occupancy_g(int group) {
  return group == 64 ? dm_occupancy_t<BF16, NT8, 1, KG, WB>() : dm_occupancy_t<BF16, NT8, 2, KG, WB>();
}

template <bool BF16, int NT8, int WB>
static int dm_occupancy_k(int group, int kgroups) {
  switch (kgroups) {
    case 1: return dm_occupancy_g<BF16, NT8, 1, WB>(group);
    case 2: return dm_occupancy_g<BF16, NT8, 2, WB>(group);
    case 4:
      if constexpr (WB == 4) return dm_occupancy_g<BF16, NT8, 4, WB>(group);
      return 1;
    default: return 1;
  }
}

template <int WB>
int dm_ctas_per_sm_wb(bool bf16, int M, int group, int kgroups) {
  switch (decode_mma_nt8(M)) {
    case 1: return bf16 ? dm_occupancy_k<true, 1, WB>(group, kgroups) : dm_occupancy_k<false, 1, WB>(group, kgroups);
    case 2: return bf16 ? dm_occupancy_k<true, 2, WB>(group, kgroups) : dm_occupancy_k<false, 2, WB>(group, kgroups);
    default: return 1;
  }
}


// Whether clusters of S CTAs (1..16) of the cluster-mode instantiation can
// be resident at all; computed once per (device, S).
template <bool BF16, int NT8, int GS, int KG, int WB>
static bool dm_cluster_fits_t(int S) {
  static std::once_flag once[kMaxOptinDevices][17];
  static bool fits[kMaxOptinDevices][17];
  constexpr int SMEM = DmGeom<NT8, KG, true, WB>::SMEM + DM_RECV_MAX;   // the largest launch
  int dev = 0;
  if (S < 1 || S > 16 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxOptinDevices) return false;
  std::call_once(once[dev][S], [&] {
    fits[dev][S] = false;
    if (cluster_optin<decode_mma_kernel<BF16, NT8, GS, true, KG, WB>>(SMEM) != cudaSuccess) return;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, S);
    cfg.blockDim = dim3(128 * KG + 32);
    cfg.dynamicSmemBytes = static_cast<size_t>(SMEM);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 1;
    attr.val.clusterDim.y = S;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    fits[dev][S] = cudaOccupancyMaxActiveClusters(&n, decode_mma_kernel<BF16, NT8, GS, true, KG, WB>, &cfg) ==
                       cudaSuccess &&
                   n > 0;
    (void)cudaGetLastError();
  });
  return fits[dev][S];
}

template <bool BF16, int NT8, int WB>
static bool dm_cluster_fits_g(int group, int kgroups, int S) {
  if (kgroups == 2)
    return group == 64 ? dm_cluster_fits_t<BF16, NT8, 1, 2, WB>(S) : dm_cluster_fits_t<BF16, NT8, 2, 2, WB>(S);
  return group == 64 ? dm_cluster_fits_t<BF16, NT8, 1, 1, WB>(S) : dm_cluster_fits_t<BF16, NT8, 2, 1, WB>(S);
}

template <int WB>
int dm_cluster_split_wb(bool bf16, int M, int K, int group, int kgroups, int requested, int *kb_per_split) {
  const int KB = K / 64, GS = group / 64;
  // rank 0 receives (S - 1) M 128 fp32 sums: at most DM_RECV_MAX bytes
  const int s_max = std::min(16, 1 + DM_RECV_MAX / (std::max(M, 1) * TILE_N * 4));
  const int req = std::max(1, std::min(requested, s_max));
  int per = (KB + req - 1) / req;
  per = (per + GS - 1) / GS * GS;
  const int S = (KB + per - 1) / per;
  bool fits = false;
  switch (decode_mma_nt8(M)) {
    case 1:
      fits = bf16 ? dm_cluster_fits_g<true, 1, WB>(group, kgroups, S)
                  : dm_cluster_fits_g<false, 1, WB>(group, kgroups, S);
      break;
    case 2:
      fits = bf16 ? dm_cluster_fits_g<true, 2, WB>(group, kgroups, S)
                  : dm_cluster_fits_g<false, 2, WB>(group, kgroups, S);
      break;
    default: break;
  }
  if (!fits) return 0;
  *kb_per_split = per;
  return S;
}

template <int WB>
cudaError_t dm_launch_wb(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int kgroups, int grid, int cluster,
                         cudaStream_t st) {
  switch (decode_mma_nt8(a.M)) {
    case 1:
      return bf16 ? launch_dm_k<true, 1, WB>(a, tmap_a, kgroups, grid, cluster, st)
                  : launch_dm_k<false, 1, WB>(a, tmap_a, kgroups, grid, cluster, st);
    case 2:
      return bf16 ? launch_dm_k<true, 2, WB>(a, tmap_a, kgroups, grid, cluster, st)
                  : launch_dm_k<false, 2, WB>(a, tmap_a, kgroups, grid, cluster, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tmw4

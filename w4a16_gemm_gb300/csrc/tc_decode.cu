// tc_decode.cu -- W4A16 GEMM for small row counts (decode) on the tcgen05
// tensor cores.
//
// With few rows of activations there is little work per weight byte, so the
// kernel must keep HBM busy rather than the tensor pipe.  Three measured
// GB300 costs shape it:
//   * one thread can issue a 64-K block (4 MMAs of M=128, N<=64, K=16 plus
//     a commit) only every ~250-400 cycles, whatever N is, while issuers in
//     different warps proceed in parallel.  Each dequant warpgroup therefore
//     has its own MMA-issuing warp and its own fp32 accumulator in TMEM; the
//     epilogue adds the accumulators in a fixed order;
//   * a bulk copy costs its issuing thread hundreds of cycles whatever its
//     size, so weights move in stages of WKB = 4 packed blocks (16 KB, one
//     copy, plus one copy each for the stage's scales and zeros) and
//     activations in 4-block boxes of a 3-D tensor map;
//   * per-thread 128-bit global loads of the weights crowd the SM's
//     memory-instruction queue that tcgen05 and mbarrier instructions also
//     use, so weights go through shared memory, and a weight stage is
//     released as soon as its dequant warps have read it, whatever the MMAs
//     are doing.
// The packed block is already in the order the consumer needs (the pages'
// fragment-order repack, "Efficient Mixed-Precision Large Language Model
// Inference with TurboMind", pith.science review, Figures 6/7): the thread that
// owns weight column r (= TMEM lane r) reads its 32 bytes of a 64-K block
// with two 128-bit shared-memory loads.
//
//   warp 0          weight producer (stage ring of WST)
//   warp 1          TMEM allocator; activation producer
//   warps 2..       one MMA-issuing warp per dequant warpgroup
//   then            DQ_WG dequant warpgroups; stage j goes to warpgroup
//                   j % DQ_WG: read each block, release the stage after its
//                   last block, dequantize exactly (w = T(s*(q-z))),
//                   tcgen05.st into one of the warpgroup's TMEM A slots; then
//                   the epilogue
//
// Parity waits stay at most one phase ahead (no aliasing) because every ring
// slot always serves the same warpgroup (WST % DQ_WG == 0 for the weight
// ring; private activation stages and TMEM slots per warpgroup), whose
// waiters have seen the slot's previous phase; copies may land out of order
// across slots.
#include <cstdint>
#include <cuda.h>

#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tc_epilogue.cuh"

namespace tmw4 {

// Debug builds count barrier polls per wait site into the trace buffer.
#ifdef TMW4_TRACE
#define TMW4_SPIN(site)                                                                       \
  (p.trace != nullptr ? reinterpret_cast<unsigned long long *>(p.trace + 15 * 256) + 2 * (site) \
                      : nullptr)
#else
#define TMW4_SPIN(site) nullptr
#endif

namespace {

constexpr int DBLOCK_N = 128;
constexpr int DBLOCK_K = 64;
constexpr int DSLOT_COLS = DBLOCK_K / 2;   // 32 TMEM columns of packed pairs per block
constexpr int WKB = 4;                     // 64-K blocks per weight / activation stage
constexpr int WST = 4;                     // weight ring depth (divisible by 1, 2, 4)
constexpr int MAX_G = WKB;                 // groups a stage can touch (group >= 64)
constexpr int W_SC_OFF = WKB * BLOCK_BYTES;                       // scales of the stage's groups
constexpr int W_ZP_OFF = W_SC_OFF + MAX_G * 2 * DBLOCK_N;         // packed zeros
constexpr int W_STAGE_BYTES = W_ZP_OFF + MAX_G * (DBLOCK_N / 2);  // 17664, a multiple of 16

// TMEM: DQ_WG accumulators of dec_dcols columns, then DQ_WG * TSW A slots.
// Up to two warpgroups share 256 columns so that two CTAs fit on an SM.
__host__ __device__ constexpr int dec_tmem_cols(int dq_wg) { return dq_wg <= 2 ? 256 : 512; }
__host__ __device__ constexpr int dec_dcols(int block_m) { return block_m < 32 ? 32 : block_m; }
// TMEM A slots per warpgroup
__host__ __device__ constexpr int dec_tsw(int block_m, int dq_wg) {
  return (dec_tmem_cols(dq_wg) / dq_wg - dec_dcols(block_m)) / DSLOT_COLS;
}
// activation stages (WKB tiles each) per warpgroup: double-buffered when the
// tiles are small, single otherwise, so that two CTAs fit on an SM
__host__ __device__ constexpr int dec_asw(int block_m, int dq_wg) {
  return block_m * dq_wg <= 32 ? 2 : 1;
}
__host__ __device__ constexpr int dec_threads(int dq_wg) { return 64 + 32 * dq_wg + 128 * dq_wg; }
__host__ __device__ constexpr int dec_a_bytes(int block_m) { return block_m * DBLOCK_K * 2; }
__host__ __device__ constexpr size_t dec_smem_bytes(int block_m, int dq_wg) {
  return 1024 +
         static_cast<size_t>(dq_wg * dec_asw(block_m, dq_wg)) * WKB * dec_a_bytes(block_m) +
         static_cast<size_t>(WST) * W_STAGE_BYTES + 1024;
}

}  // namespace

template <bool BF16, int BLOCK_M, int DQ_WG>
__global__ void __launch_bounds__(dec_threads(DQ_WG), DQ_WG <= 2 ? 2 : 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs p) {
  constexpr int TSW = dec_tsw(BLOCK_M, DQ_WG);
  constexpr int TSLOTS = DQ_WG * TSW;
  constexpr int ASW = dec_asw(BLOCK_M, DQ_WG);
  constexpr int ASTAGES = DQ_WG * ASW;
  constexpr int TCOLS = dec_tmem_cols(DQ_WG);
  constexpr int A_KB = dec_a_bytes(BLOCK_M);
  constexpr int A_STAGE = WKB * A_KB;
  constexpr int DCOLS = dec_dcols(BLOCK_M);
  constexpr int A_COL0 = DQ_WG * DCOLS;
  constexpr int FIRST_DQ_WARP = 2 + DQ_WG;
  constexpr uint32_t IDESC = idesc_f16(BF16 ? 1u : 0u, 128u, static_cast<uint32_t>(BLOCK_M));
  static_assert(BLOCK_M == 16 || BLOCK_M == 32 || BLOCK_M == 64, "decode tiles");
  static_assert(TSW >= 2, "each warpgroup needs two TMEM A slots to overlap dequant and MMA");
  static_assert(A_COL0 + TSLOTS * DSLOT_COLS <= TCOLS, "TMEM budget");
  static_assert(WST % DQ_WG == 0, "weight ring: a stage must always go to the same warpgroup");
  static_assert(A_KB % 1024 == 0, "swizzle atoms");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;                                   // [ASTAGES][WKB][BLOCK_M x 128 B]
  uint8_t *sW = sA + ASTAGES * A_STAGE;                 // [WST][W_STAGE_BYTES]
  uint64_t *wfull_bar = reinterpret_cast<uint64_t *>(sW + WST * W_STAGE_BYTES);  // stage landed
  uint64_t *wempty_bar = wfull_bar + WST;               // stage read by its 4 dequant warps
  uint64_t *afull_bar = wempty_bar + WST;               // activation stage landed
  uint64_t *aempty_bar = afull_bar + ASTAGES;           // MMAs reading it retired
  uint64_t *tfull_bar = aempty_bar + ASTAGES;           // dequantized block in TMEM
  uint64_t *kfree_bar = tfull_bar + TSLOTS;             // MMAs of the slot's block retired
  uint64_t *accum_bar = kfree_bar + TSLOTS;             // every issuer's MMAs retired
  uint64_t *drain_bar = accum_bar + 1;                  // [DQ_WG] abort path
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain_bar + DQ_WG);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  int *last_flag = reinterpret_cast<int *>(tmem_holder + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x;
  const int n0 = nt * DBLOCK_N;
  const int m0 = blockIdx.y * BLOCK_M;
  const int split = blockIdx.z;
  const int KB = p.K / DBLOCK_K;
  const int G_rows = p.K / p.group;
  const int kb0 = split * p.kb_per_split;
  const int nkb = max(0, min(KB, kb0 + p.kb_per_split) - kb0);
  const int nst = (nkb + WKB - 1) / WKB;                // stages of this CTA
  const int nacc = min(DQ_WG, nst);                     // warpgroups that own a stage

  if (threadIdx.x == 0) {
    TMW4_STAMP(7, 1);
    for (int s = 0; s < WST; ++s) {
      mbar_init(wfull_bar + s, 1);
      mbar_init(wempty_bar + s, 4);
    }
    for (int s = 0; s < ASTAGES; ++s) {
      mbar_init(afull_bar + s, 1);
      mbar_init(aempty_bar + s, 1);
    }
    for (int s = 0; s < TSLOTS; ++s) {
      mbar_init(tfull_bar + s, 4);
      mbar_init(kfree_bar + s, 1);
    }
    mbar_init(accum_bar, nacc > 0 ? nacc : 1);
    for (int g = 0; g < DQ_WG; ++g) mbar_init(drain_bar + g, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmap_a);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  if (threadIdx.x == 0) TMW4_STAMP(7, 0);

  if (warp == 0) {
    // --------------------------------------------------- weight producer
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nst; ++j) {
        const int s = j % WST;
        if (j >= WST && !mbar_wait_bounded(wempty_bar + s, ((j / WST) & 1) ^ 1u, p.limit_ns,
                                           abort_flag, p.err, SITE_PRODUCER_EMPTY, j, TMW4_SPIN(0)))
          break;
        const int kbf = kb0 + j * WKB;
        const int nb = min(WKB, nkb - j * WKB);
        const int gf = (kbf * DBLOCK_K) / p.group;
        const int ng = ((kbf + nb) * DBLOCK_K - 1) / p.group - gf + 1;
        uint8_t *st = sW + s * W_STAGE_BYTES;
        const uint32_t tx = nb * BLOCK_BYTES + ng * 2 * DBLOCK_N +
                            (p.zeros != nullptr ? ng * (DBLOCK_N / 2) : 0);
        mbar_arrive_expect_tx(wfull_bar + s, tx);
        tma_bulk_g2s(st, p.qw + (static_cast<size_t>(nt) * KB + kbf) * BLOCK_BYTES,
                     nb * BLOCK_BYTES, wfull_bar + s);
        tma_bulk_g2s(st + W_SC_OFF, p.scales + (static_cast<size_t>(nt) * G_rows + gf) * DBLOCK_N,
                     ng * 2 * DBLOCK_N, wfull_bar + s);
        if (p.zeros != nullptr)
          tma_bulk_g2s(st + W_ZP_OFF,
                       p.zeros + (static_cast<size_t>(nt) * G_rows + gf) * (DBLOCK_N / 2),
                       ng * (DBLOCK_N / 2), wfull_bar + s);
        TMW4_STAMP(0, j);
        issued = j + 1;
      }
      // every copy issued must have landed before the CTA exits
      for (int s = 0; s < WST && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / WST) * WST;
        mbar_wait_bounded(wfull_bar + s, (last / WST) & 1, p.limit_ns, nullptr, p.err,
                          SITE_DRAIN_TMA, last);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------- activation producer
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nst; ++j) {
        const int cs = j / DQ_WG;                        // j is stage cs of warpgroup j % DQ_WG
        const int s = (j % DQ_WG) * ASW + cs % ASW;
        if (cs >= ASW && !mbar_wait_bounded(aempty_bar + s, ((cs / ASW) & 1) ^ 1u, p.limit_ns,
                                            abort_flag, p.err, SITE_PRODUCER_EMPTY, j, TMW4_SPIN(1)))
          break;
        const int kbf = kb0 + j * WKB;
        const int nb = min(WKB, nkb - j * WKB);
        uint8_t *dst = sA + s * A_STAGE;
        if (p.act_map_3d) {
          // a box of WKB tiles; tiles past the end of K are zero-filled and
          // still counted by the transaction
          mbar_arrive_expect_tx(afull_bar + s, A_STAGE);
          tma_load_3d(dst, &tmap_a, 0, m0, kbf, afull_bar + s);
        } else {
          mbar_arrive_expect_tx(afull_bar + s, nb * A_KB);
          for (int b = 0; b < nb; ++b)
            tma_load_2d(dst + b * A_KB, &tmap_a, (kbf + b) * DBLOCK_K, m0, afull_bar + s);
        }
        issued = j + 1;
      }
      for (int j = max(0, issued - ASTAGES); j < issued; ++j) {
        const int cs = j / DQ_WG;
        mbar_wait_bounded(afull_bar + (j % DQ_WG) * ASW + cs % ASW, (cs / ASW) & 1, p.limit_ns,
                          nullptr, p.err, SITE_DRAIN_TMA, j);
      }
    }
  } else if (warp < FIRST_DQ_WARP) {
    // ---------------------------------- MMA issue for warpgroup warp - 2
    const int wg = warp - 2;
    if (lane == 0) {
      bool ok = true, any = false;
      const uint32_t d_tmem = tmem + wg * DCOLS;
      const uint64_t desc0 = smem_desc_k128(smem_u32(sA));
      int c = 0;                                         // this warpgroup's block counter
      for (int j = wg, cs = 0; j < nst && ok; j += DQ_WG, ++cs) {
        const int as = wg * ASW + cs % ASW;
        if (!mbar_wait_bounded(afull_bar + as, (cs / ASW) & 1, p.limit_ns, abort_flag, p.err,
                               SITE_MMA_FULL, j, TMW4_SPIN(2))) {
          ok = false;
          break;
        }
        const int nb = min(WKB, nkb - j * WKB);
        for (int b = 0; b < nb; ++b, ++c) {
          const int s = wg * TSW + c % TSW;
          const int i = j * WKB + b;
          TMW4_STAMP(8, i);
          if (!mbar_wait_bounded(tfull_bar + s, (c / TSW) & 1, p.limit_ns, abort_flag, p.err,
                                 SITE_MMA_AFULL, i, TMW4_SPIN(3))) {
            ok = false;
            break;
          }
          tc_fence_after();
          TMW4_STAMP(4, i);
          tc_mma_ts_kblock(d_tmem, tmem + A_COL0 + s * DSLOT_COLS,
                           desc0 + static_cast<uint64_t>((as * A_STAGE + b * A_KB) >> 4), IDESC,
                           c == 0 ? 1u : 0u);
          any = true;
          TMW4_STAMP(9, i);
          tc_commit(kfree_bar + s);
          TMW4_STAMP(5, i);
        }
        if (ok) tc_commit(aempty_bar + as);
      }
      if (ok && any) {
        tc_commit(accum_bar);
      } else if (any) {
        tc_commit(drain_bar + wg);
        mbar_wait_bounded(drain_bar + wg, 0, p.limit_ns, nullptr, p.err, SITE_DRAIN_MMA, wg);
      }
    }
  } else {
    // ------------------------------------------------- dequant + epilogue
    const int dw = warp - FIRST_DQ_WARP;
    const int wg = dw >> 2;
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;            // weight column within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int w_off = (r >> 6) * ATOM_BYTES + (r & 63) * 16;
    const int zshift = (r & 1) * 4;
    bool ok = true;
    int c = 0;
    for (int j = wg; j < nst && ok; j += DQ_WG) {
      const int ws = j % WST;
      if (!mbar_wait_warp(wfull_bar + ws, (j / WST) & 1, p.limit_ns, abort_flag, p.err,
                          SITE_DQ_FULL, j, TMW4_SPIN(4))) {
        ok = false;
        break;
      }
      const uint8_t *st = sW + ws * W_STAGE_BYTES;
      const int kbf = kb0 + j * WKB;
      const int nb = min(WKB, nkb - j * WKB);
      const int gf = (kbf * DBLOCK_K) / p.group;
      for (int b = 0; b < nb; ++b, ++c) {
        const int i = j * WKB + b;
        const int ts = wg * TSW + c % TSW;
        if (quarter == 2 && lane == 0) TMW4_STAMP(12, i);
        const uint4 v0 = *reinterpret_cast<const uint4 *>(st + b * BLOCK_BYTES + w_off);
        const uint4 v1 = *reinterpret_cast<const uint4 *>(st + b * BLOCK_BYTES + w_off + 1024);
        const int gi = ((kbf + b) * DBLOCK_K) / p.group - gf;
        const uint16_t sc = reinterpret_cast<const uint16_t *>(st + W_SC_OFF)[gi * DBLOCK_N + r];
        const uint32_t z =
            p.zeros != nullptr
                ? (static_cast<uint32_t>(st[W_ZP_OFF + gi * (DBLOCK_N / 2) + (r >> 1)]) >> zshift) & 0xFu
                : 8u;
        if (b == nb - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(wempty_bar + ws);   // this warp is done with the stage
        }
        if (c >= TSW && !mbar_wait_warp(kfree_bar + ts, ((c / TSW) & 1) ^ 1u, p.limit_ns,
                                        abort_flag, p.err, SITE_DQ_AEMPTY, i, TMW4_SPIN(5))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (quarter == 2 && lane == 0) TMW4_STAMP(2, i);
        const uint32_t s2 = dup16(sc), zm2 = zero_magic2<BF16>(z);
        uint32_t d0[16], d1[16];
        {
          const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
          const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t o[4];
            dequant_word<BF16>(w0[q4], zm2, s2, o);
#pragma unroll
            for (int q = 0; q < 4; ++q) d0[4 * q4 + q] = o[q];
            dequant_word<BF16>(w1[q4], zm2, s2, o);
#pragma unroll
            for (int q = 0; q < 4; ++q) d1[4 * q4 + q] = o[q];
          }
        }
        __syncwarp();
        const uint32_t ta = tmem + lane_addr + A_COL0 + ts * DSLOT_COLS;
        tmem_st_16(ta, d0);
        tmem_st_16(ta + 16, d1);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tfull_bar + ts);
        if (quarter == 2 && lane == 0) TMW4_STAMP(3, i);
      }
    }
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (ok && nkb > 0)
      ok = mbar_wait_warp(accum_bar, 0, p.limit_ns, abort_flag, p.err, SITE_EPI_ACCUM, 0, TMW4_SPIN(6));
    tc_fence_after();
    if (dw == 0 && lane == 0) TMW4_STAMP(6, 0);
    tc_epilogue<BF16, BLOCK_M, DQ_WG>(p, tmem + lane_addr, wg, dw, lane, r, n0, m0, split, ok, nacc,
                                      static_cast<uint32_t>(DCOLS), last_flag);
    if (dw == 0 && lane == 0) TMW4_STAMP(6, 1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TCOLS);
  }
}

bool tc_decode_ok(int block_m, int dq_warps) {
  if (block_m != 16 && block_m != 32 && block_m != 64) return false;
  if (dq_warps != 4 && dq_warps != 8 && dq_warps != 16) return false;
  const int wg = dq_warps / 4;
  return dec_tsw(block_m, wg) >= 2 && WST % wg == 0;
}

int tc_decode_slots(int block_m, int dq_warps) { return dec_tsw(block_m, dq_warps / 4); }

int tc_decode_kblocks_per_stage() { return WKB; }

template <bool BF16, int BLOCK_M, int DQ_WG>
static cudaError_t launch_dec_t(const GemmArgs &a, const CUtensorMap &tmap, cudaStream_t st) {
  auto kern = tc_decode_kernel<BF16, BLOCK_M, DQ_WG>;
  const size_t smem = dec_smem_bytes(BLOCK_M, DQ_WG);
  static int attr_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_device != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_device = dev;
  }
  dim3 grid(a.N / DBLOCK_N, (a.M + BLOCK_M - 1) / BLOCK_M, a.splits);
  kern<<<grid, dec_threads(DQ_WG), smem, st>>>(tmap, a);
  return cudaGetLastError();
}

template <bool BF16, int BLOCK_M>
static cudaError_t launch_dec_bm(const GemmArgs &a, const CUtensorMap &tmap, int dq, cudaStream_t st) {
  switch (dq) {
    case 4: return launch_dec_t<BF16, BLOCK_M, 1>(a, tmap, st);
    case 8: return launch_dec_t<BF16, BLOCK_M, 2>(a, tmap, st);
    case 16: return launch_dec_t<BF16, BLOCK_M, 4>(a, tmap, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_tc_decode(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int block_m,
                             int dq_warps, cudaStream_t st) {
  switch (block_m) {
    case 16: return bf16 ? launch_dec_bm<true, 16>(a, tmap_a, dq_warps, st)
                         : launch_dec_bm<false, 16>(a, tmap_a, dq_warps, st);
    case 32: return bf16 ? launch_dec_bm<true, 32>(a, tmap_a, dq_warps, st)
                         : launch_dec_bm<false, 32>(a, tmap_a, dq_warps, st);
    case 64: return bf16 ? launch_dec_bm<true, 64>(a, tmap_a, dq_warps, st)
                         : launch_dec_bm<false, 64>(a, tmap_a, dq_warps, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tmw4

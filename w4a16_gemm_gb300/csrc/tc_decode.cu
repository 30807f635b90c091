// tc_decode.cu -- W4A16 GEMM for small row counts (decode): a persistent,
// stream-K tcgen05 kernel.
//
// With few rows of activations there is little work per weight byte, so the
// kernel must keep HBM busy rather than the tensor pipe.  Measured GB300 costs
// shape it:
//   * one thread can issue a 64-K block (4 MMAs of M=128, N<=64, K=16 plus
//     a commit) only every ~250-400 cycles, whatever N is, while issuers in
//     different warps proceed in parallel.  Each dequant warpgroup therefore
//     has its own MMA-issuing warp and its own fp32 accumulators in TMEM;
//   * a bulk copy costs its issuing thread hundreds of cycles whatever its
//     size, so weights move in stages of WKB = 4 packed blocks (16 KB, one
//     copy, plus one copy each for the stage's scales and zeros) and
//     activations in 4-block boxes of a 3-D tensor map;
//   * per-thread 128-bit global loads of the weights crowd the SM's
//     memory-instruction queue that tcgen05 and mbarrier instructions also
//     use, so weights go through shared memory; a weight stage is released
//     once its dequant warps have used its data;
//   * a weight stage takes ~1.5-2 us from copy issue to arrival under load,
//     so each warpgroup keeps several stages in flight: one CTA per SM with a
//     deep ring;
//   * with one CTA per SM, whole-tile CTAs leave SMs idle (e.g. 224 tiles on
//     152 SMs), so the work is split stream-K style: the (tile, 16 KB stage)
//     units of the problem are divided evenly over a persistent grid, a CTA
//     runs its units in order, and a tile cut between CTAs is finished by the
//     last one to arrive, which adds the fp32 partials in a fixed order.
// The packed block is already in the order the consumer needs (the pages'
// fragment-order repack, "Efficient Mixed-Precision Large Language Model
// Inference with TurboMind", pith.science review, Figures 6/7): the thread that
// owns weight column r (= TMEM lane r) reads its 32 bytes of a 64-K block
// with two 128-bit shared-memory loads.
//
//   warp 0          weight producer (stage ring of WST)
//   warp 1          TMEM allocator; activation producer
//   warps 2..       one MMA-issuing warp per dequant warpgroup
//   next 4 warps    epilogue warpgroup: per tile segment, waits for the
//                   accumulators, adds them, writes C or an fp32 partial
//   then            DQ_WG dequant warpgroups; the CTA's j-th stage goes to
//                   warpgroup j % DQ_WG, which dequantizes exactly
//                   (w = T(s*(q-z))) two blocks at a time into its TMEM A slots
//
// Each warpgroup has two accumulators and alternates between them from one
// tile segment to the next, so the MMAs of a segment overlap the epilogue of
// the previous one.
//
// Parity waits stay at most one phase ahead (no aliasing) because every ring
// slot always serves the same warpgroup (WST % DQ_WG == 0 for the weight
// ring; private activation stages, TMEM slots and accumulators per
// warpgroup), whose waiters have seen the slot's previous phase, and because
// one thread's tcgen05 commits complete in issue order; copies may land out
// of order across slots.
#include <algorithm>
#include <cstdint>
#include <cuda.h>

#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tc_epilogue.cuh"

namespace tmw4 {

// Debug builds with TMW4_SPIN_COUNT count barrier polls per wait site into
// the trace buffer (global atomics: they slow the kernel down).
#if defined(TMW4_TRACE) && defined(TMW4_SPIN_COUNT)
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
constexpr int MAX_G = WKB;                 // groups a stage can touch (group >= 64)
constexpr int W_SC_OFF = WKB * BLOCK_BYTES;                       // scales of the stage's groups
constexpr int W_ZP_OFF = W_SC_OFF + MAX_G * 2 * DBLOCK_N;         // packed zeros
constexpr int W_STAGE_BYTES = W_ZP_OFF + MAX_G * (DBLOCK_N / 2);  // 17664, a multiple of 16
constexpr int TMEM_COLS = 512;             // one CTA per SM
constexpr long long SMEM_BUDGET = 220 * 1024;

__host__ __device__ constexpr int dec_dcols(int block_m) { return block_m < 32 ? 32 : block_m; }
// TMEM columns per warpgroup: two accumulators, then the A slots (at most 8)
__host__ __device__ constexpr int dec_wg_cols(int dq_wg) { return (TMEM_COLS / dq_wg) / 32 * 32; }
__host__ __device__ constexpr int dec_tsw_fit(int block_m, int dq_wg) {
  return (dec_wg_cols(dq_wg) - 2 * dec_dcols(block_m)) / DSLOT_COLS;
}
// a power of two (ring indices are masks and shifts), at most 8
__host__ __device__ constexpr int dec_tsw(int block_m, int dq_wg) {
  return dec_tsw_fit(block_m, dq_wg) >= 8   ? 8
         : dec_tsw_fit(block_m, dq_wg) >= 4 ? 4
         : dec_tsw_fit(block_m, dq_wg) >= 2 ? 2
                                            : 1;
}
__host__ __device__ constexpr long long dec_a_stage(int block_m) {
  return static_cast<long long>(WKB) * block_m * DBLOCK_K * 2;
}
// activation stages per warpgroup: double-buffered when it leaves room for a
// weight ring of six stages
__host__ __device__ constexpr int dec_asw(int block_m, int dq_wg) {
  return 2 * dq_wg * dec_a_stage(block_m) + 6 * W_STAGE_BYTES <= SMEM_BUDGET ? 2 : 1;
}
// weight ring depth: the deepest multiple of dq_wg (at most 12) that fits
__host__ __device__ constexpr int dec_wst_fit(int block_m, int dq_wg) {
  return static_cast<int>(
      ((SMEM_BUDGET - dq_wg * dec_asw(block_m, dq_wg) * dec_a_stage(block_m)) / W_STAGE_BYTES) /
      dq_wg * dq_wg);
}
__host__ __device__ constexpr int dec_wst(int block_m, int dq_wg) {
  return dec_wst_fit(block_m, dq_wg) > 12 ? 12 / dq_wg * dq_wg : dec_wst_fit(block_m, dq_wg);
}
__host__ __device__ constexpr int dec_threads(int dq_wg) { return 64 + 32 * dq_wg + 128 + 128 * dq_wg; }
__host__ __device__ constexpr long long dec_smem_bytes(int block_m, int dq_wg) {
  return 1024 + dq_wg * dec_asw(block_m, dq_wg) * dec_a_stage(block_m) +
         static_cast<long long>(dec_wst(block_m, dq_wg)) * W_STAGE_BYTES + 1024;
}

// Position of a unit: tile t (= mt * NT + nt) and stage s of that tile.
// Loops step it forward instead of dividing a 64-bit unit index: a 64-bit
// division by a runtime value costs a few hundred cycles per loop trip.
struct UnitPos {
  int t, s, mt, nt;
  __device__ __forceinline__ void step(int n, int S, int NT) {
    s += n;
    while (s >= S) {
      s -= S;
      ++t;
      if (++nt == NT) {
        nt = 0;
        ++mt;
      }
    }
  }
};

}  // namespace

template <bool BF16, int BLOCK_M, int DQ_WG>
__global__ void __launch_bounds__(dec_threads(DQ_WG), 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs p) {
  constexpr int TSW = dec_tsw(BLOCK_M, DQ_WG);
  constexpr int TSLOTS = DQ_WG * TSW;
  constexpr int ASW = dec_asw(BLOCK_M, DQ_WG);
  constexpr int ASTAGES = DQ_WG * ASW;
  constexpr int WST = dec_wst(BLOCK_M, DQ_WG);
  constexpr int A_KB = BLOCK_M * DBLOCK_K * 2;
  constexpr int A_STAGE = static_cast<int>(dec_a_stage(BLOCK_M));
  constexpr int DCOLS = dec_dcols(BLOCK_M);
  constexpr int WG_COLS = dec_wg_cols(DQ_WG);
  constexpr int ISSUE_WARP0 = 2;
  constexpr int EPI_WARP0 = 2 + DQ_WG;
  constexpr int DQ_WARP0 = EPI_WARP0 + 4;
  constexpr uint32_t IDESC = idesc_f16(BF16 ? 1u : 0u, 128u, static_cast<uint32_t>(BLOCK_M));
  static_assert(BLOCK_M == 16 || BLOCK_M == 32 || BLOCK_M == 64, "decode tiles");
  static_assert(TSW >= 2, "a warpgroup needs two TMEM A slots (one block pair)");
  static_assert(WST >= 2 * DQ_WG && WST % DQ_WG == 0, "weight ring");
  static_assert(A_KB % 1024 == 0, "swizzle atoms");
  static_assert(dec_smem_bytes(BLOCK_M, DQ_WG) <= 227 * 1024, "shared memory");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align_smem_1024(smem_raw);
  uint8_t *sA = smem;                                   // [ASTAGES][WKB][BLOCK_M x 128 B]
  uint8_t *sW = sA + ASTAGES * A_STAGE;                 // [WST][W_STAGE_BYTES]
  uint64_t *wfull_bar = reinterpret_cast<uint64_t *>(sW + WST * W_STAGE_BYTES);  // stage landed
  uint64_t *wempty_bar = wfull_bar + WST;               // stage read by its 4 dequant warps
  uint64_t *afull_bar = wempty_bar + WST;               // activation stage landed
  uint64_t *aempty_bar = afull_bar + ASTAGES;           // MMAs reading it retired
  uint64_t *tfull_bar = aempty_bar + ASTAGES;           // dequantized block in TMEM
  uint64_t *kfree_bar = tfull_bar + TSLOTS;             // MMAs of the slot's block retired
  uint64_t *accfull_bar = kfree_bar + TSLOTS;           // [DQ_WG][2] segment's MMAs retired
  uint64_t *accempty_bar = accfull_bar + 2 * DQ_WG;     // [DQ_WG][2] epilogue has read it
  uint64_t *drain_bar = accempty_bar + 2 * DQ_WG;       // [DQ_WG] abort path
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain_bar + DQ_WG);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  int *last_flag = reinterpret_cast<int *>(tmem_holder + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = p.K / DBLOCK_K;
  const int S = (KB + WKB - 1) / WKB;                   // stages per tile
  const int NT = p.N / DBLOCK_N;
  const long long T = static_cast<long long>(NT) * ((p.M + BLOCK_M - 1) / BLOCK_M);
  const long long U = T * S;
  const long long G = gridDim.x;
  const long long u0 = unit_begin(blockIdx.x, U, G);
  const int nloc = static_cast<int>(unit_begin(blockIdx.x + 1, U, G) - u0);
  const int G_rows = p.K / p.group;
  const int gshift = p.group == 128 ? 1 : 0;            // 64-K blocks per group: 1 << gshift
  UnitPos pos0;                                         // this CTA's first unit
  pos0.t = static_cast<int>(u0 / S);
  pos0.s = static_cast<int>(u0 - static_cast<long long>(pos0.t) * S);
  pos0.mt = pos0.t / NT;
  pos0.nt = pos0.t - pos0.mt * NT;

  if (threadIdx.x == 0) {
    TMW4_STAMP(7, 1);
#ifdef TMW4_TRACE
    if (p.trace != nullptr && blockIdx.x < 256)
      p.trace[13 * 256 + blockIdx.x] = static_cast<long long>(globaltimer_ns());
#endif
    *abort_flag = 0;
    *last_flag = 0;
    prefetch_tensormap(&tmap_a);
  }
  {
    // one barrier per thread: the barriers are contiguous, in the order
    // wfull, wempty, afull, aempty, tfull, kfree, accfull, accempty, drain
    constexpr int NBAR = 2 * WST + 2 * ASTAGES + 2 * TSLOTS + 4 * DQ_WG + DQ_WG;
    static_assert(NBAR <= 64 + 32 * DQ_WG + 128 + 128 * DQ_WG, "one thread per barrier");
    const int b = threadIdx.x;
    if (b < NBAR) {
      int cnt = 1;
      if (b >= WST && b < 2 * WST) cnt = 4;                                   // wempty
      const int t0 = 2 * WST + 2 * ASTAGES;
      if (b >= t0 && b < t0 + TSLOTS) cnt = 4;                                 // tfull
      const int e0 = t0 + 2 * TSLOTS + 2 * DQ_WG;
      if (b >= e0 && b < e0 + 2 * DQ_WG) cnt = 4;                              // accempty
      mbar_init(wfull_bar + b, cnt);
      fence_mbar_init();
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  __syncwarp();   // threads that initialised a barrier rejoin their warp first
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  if (threadIdx.x == 0) TMW4_STAMP(7, 0);
  // Only the activation producer and the epilogue touch memory that an
  // earlier kernel in the stream may write (A; C, the partials and the
  // counters): they call pdl_wait() first.  The weight stream starts at once.
  pdl_launch_dependents();

  if (warp == 0) {
    // --------------------------------------------------- weight producer
    if (lane == 0) {
      int issued = 0;
      UnitPos pos = pos0;
      for (int j = 0; j < nloc; ++j, pos.step(1, S, NT)) {
        const int s = j % WST;
        if (j >= WST && !mbar_wait_idle(wempty_bar + s, ((j / WST) & 1) ^ 1u, p.limit_ns,
                                        abort_flag, p.err, SITE_PRODUCER_EMPTY, j))
          break;
        const int nt = pos.nt;
        const int kbf = pos.s * WKB;
        const int nb = min(WKB, KB - kbf);
        const int gf = kbf >> gshift;
        const int ng = ((kbf + nb - 1) >> gshift) - gf + 1;
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
      pdl_wait();
      int issued = 0;
      UnitPos pos = pos0;
      for (int j = 0; j < nloc; ++j, pos.step(1, S, NT)) {
        const int cs = j / DQ_WG;                        // j is stage cs of warpgroup j % DQ_WG
        const int s = (j % DQ_WG) * ASW + cs % ASW;
        if (cs >= ASW && !mbar_wait_idle(aempty_bar + s, ((cs / ASW) & 1) ^ 1u, p.limit_ns,
                                         abort_flag, p.err, SITE_PRODUCER_EMPTY, j))
          break;
        const int mt = pos.mt;
        const int kbf = pos.s * WKB;
        const int nb = min(WKB, KB - kbf);
        uint8_t *dst = sA + s * A_STAGE;
        if (p.act_map_3d) {
          // a box of WKB tiles; tiles past the end of K are zero-filled and
          // still counted by the transaction
          mbar_arrive_expect_tx(afull_bar + s, A_STAGE);
          tma_load_3d(dst, &tmap_a, 0, mt * BLOCK_M, kbf, afull_bar + s);
        } else {
          mbar_arrive_expect_tx(afull_bar + s, nb * A_KB);
          for (int b = 0; b < nb; ++b)
            tma_load_2d(dst + b * A_KB, &tmap_a, (kbf + b) * DBLOCK_K, mt * BLOCK_M, afull_bar + s);
        }
        TMW4_STAMP(1, j);
        issued = j + 1;
      }
      for (int j = max(0, issued - ASTAGES); j < issued; ++j) {
        const int cs = j / DQ_WG;
        mbar_wait_bounded(afull_bar + (j % DQ_WG) * ASW + cs % ASW, (cs / ASW) & 1, p.limit_ns,
                          nullptr, p.err, SITE_DRAIN_TMA, j);
      }
    }
  } else if (warp < EPI_WARP0) {
    // ------------------------------ MMA issue for warpgroup warp - ISSUE_WARP0
    const int wg = warp - ISSUE_WARP0;
    if (lane == 0) {
      bool ok = true, any = false;
      const uint32_t wg_tmem = tmem + wg * WG_COLS;
      const uint64_t desc0 = smem_desc_k128(smem_u32(sA));
      unsigned c = 0;        // this warpgroup's block counter (TMEM slot ring)
      int e = -1;       // this warpgroup's segment counter (accumulator ring)
      int t_cur = -1;
      bool first = true;
      UnitPos pos = pos0;
      pos.step(wg, S, NT);
      for (int j = wg, cs = 0; j < nloc && ok; j += DQ_WG, ++cs) {
        const int t = pos.t;
        if (t != t_cur) {
          // first stage of a new tile segment for this warpgroup
          t_cur = t;
          ++e;
          first = true;
          if (e >= 2 && !mbar_wait_bounded(accempty_bar + wg * 2 + (e & 1), ((e >> 1) & 1) ^ 1u,
                                           p.limit_ns, abort_flag, p.err, SITE_MMA_FULL, j,
                                           TMW4_SPIN(2))) {
            ok = false;
            break;
          }
        }
        const uint32_t d_tmem = wg_tmem + (e & 1) * DCOLS;
        const int as = wg * ASW + cs % ASW;
        if (!mbar_wait_bounded(afull_bar + as, (cs / ASW) & 1, p.limit_ns, abort_flag, p.err,
                               SITE_MMA_FULL, j, TMW4_SPIN(2))) {
          ok = false;
          break;
        }
        const int nb = min(WKB, KB - pos.s * WKB);
        if (nb == WKB) {
          // a full stage arrives in pairs: one wait (the pair's second block
          // is published after its first) and one fence per eight MMAs
#pragma unroll
          for (int b = 0; b < WKB; b += 2, c += 2) {
            const unsigned s0 = c & (TSW - 1), s1 = (c + 1) & (TSW - 1);
            if (!mbar_wait_bounded(tfull_bar + wg * TSW + s1, ((c + 1) / TSW) & 1u, p.limit_ns,
                                   abort_flag, p.err, SITE_MMA_AFULL, j * WKB + b, TMW4_SPIN(3))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bdesc = desc0 + static_cast<uint64_t>((as * A_STAGE + b * A_KB) >> 4);
            tc_mma_ts_kblock(d_tmem, wg_tmem + 2 * DCOLS + s0 * DSLOT_COLS, bdesc, IDESC,
                             first ? 1u : 0u);
            tc_commit(kfree_bar + wg * TSW + s0);
            tc_mma_ts_kblock(d_tmem, wg_tmem + 2 * DCOLS + s1 * DSLOT_COLS,
                             bdesc + static_cast<uint64_t>(A_KB >> 4), IDESC, 0u);
            tc_commit(kfree_bar + wg * TSW + s1);
            first = false;
            any = true;
          }
        } else
        for (int b = 0; b < nb; ++b, ++c) {
          const unsigned s = c & (TSW - 1);
          TMW4_STAMP(8, j * WKB + b);
          if (!mbar_wait_bounded(tfull_bar + wg * TSW + s, (c / TSW) & 1u, p.limit_ns, abort_flag,
                                 p.err, SITE_MMA_AFULL, j * WKB + b, TMW4_SPIN(3))) {
            ok = false;
            break;
          }
          tc_fence_after();
          TMW4_STAMP(4, j * WKB + b);
          tc_mma_ts_kblock(d_tmem, wg_tmem + 2 * DCOLS + s * DSLOT_COLS,
                           desc0 + static_cast<uint64_t>((as * A_STAGE + b * A_KB) >> 4), IDESC,
                           first ? 1u : 0u);
          first = false;
          any = true;
          tc_commit(kfree_bar + wg * TSW + s);
          TMW4_STAMP(5, j * WKB + b);
        }
        if (!ok) break;
        tc_commit(aempty_bar + as);
        // last stage of this segment for this warpgroup: hand the accumulator over
        pos.step(DQ_WG, S, NT);
        if (j + DQ_WG >= nloc || pos.t != t) tc_commit(accfull_bar + wg * 2 + (e & 1));
      }
      if (!ok && any) {
        tc_commit(drain_bar + wg);
        mbar_wait_bounded(drain_bar + wg, 0, p.limit_ns, nullptr, p.err, SITE_DRAIN_MMA, wg);
      }
    }
  } else if (warp < DQ_WARP0) {
    // -------------------------------------------------------------- epilogue
    pdl_wait();
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                 // weight column within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int M = p.M, N = p.N;
    int e_of[DQ_WG];                                   // per warpgroup: segments seen so far
#pragma unroll
    for (int w = 0; w < DQ_WG; ++w) e_of[w] = -1;
    bool ok = true;
    int jseg = 0;                                      // first local stage of the segment
    UnitPos pos = pos0;
    while (jseg < nloc && ok) {
      const int t = pos.t;
      const int s_begin = pos.s;                         // first stage of the tile in this CTA
      const int jend = min(nloc, jseg + (S - s_begin));
      const int mt = pos.mt, nt = pos.nt;
      const int m0 = mt * BLOCK_M, n = nt * DBLOCK_N + r;
      // the warpgroups with a stage in this segment, in a fixed order
      const int nwg = min(jend - jseg, DQ_WG);
      if (quarter == 0 && lane == 0) TMW4_STAMP(6, jseg);
      float acc[BLOCK_M];
#pragma unroll
      for (int x = 0; x < BLOCK_M; ++x) acc[x] = 0.f;
      for (int q = 0; q < nwg && ok; ++q) {
        const int w = (jseg + q) % DQ_WG;
        int e = 0;
#pragma unroll
        for (int ww = 0; ww < DQ_WG; ++ww)
          if (ww == w) e = ++e_of[ww];
        ok = mbar_wait_warp(accfull_bar + w * 2 + (e & 1), (e >> 1) & 1, p.limit_ns, abort_flag,
                            p.err, SITE_EPI_ACCUM, jseg, TMW4_SPIN(6));
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_addr = tmem + lane_addr + w * WG_COLS + (e & 1) * DCOLS;
#pragma unroll
        for (int c0 = 0; c0 < BLOCK_M; c0 += 16) {
          uint32_t v[16];
          tmem_ld_16(a_addr + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 16; ++x) acc[c0 + x] += __uint_as_float(v[x]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accempty_bar + w * 2 + (e & 1));
      }
      if (!ok) break;
      if (quarter == 0 && lane == 0) TMW4_STAMP(10, jseg);
      const bool whole = s_begin == 0 && jend - jseg == S;
      if (whole) {
#pragma unroll
        for (int x = 0; x < BLOCK_M; ++x)
          if (m0 + x < M) p.C[static_cast<size_t>(m0 + x) * N + n] = f32_to_16<BF16>(acc[x]);
      } else {
        // partial of contributor (this CTA) of tile t; the last to arrive sums
        const int c_first = cta_of_unit(static_cast<long long>(t) * S, U, G);
        const int c_last = cta_of_unit(static_cast<long long>(t + 1) * S - 1, U, G);
        const int ncontrib = c_last - c_first + 1;
        const int idx = static_cast<int>(blockIdx.x) - c_first;
        float *slot_base = p.ws + static_cast<size_t>(t) * p.ws_slots * (DBLOCK_N * BLOCK_M);
        float *mine = slot_base + static_cast<size_t>(idx) * (DBLOCK_N * BLOCK_M);
        // slot layout [column r][row x]: a thread's BLOCK_M values are
        // contiguous, so it writes and later reads them as 16-byte vectors
        float4 *mine4 = reinterpret_cast<float4 *>(mine + r * BLOCK_M);
#pragma unroll
        for (int x = 0; x < BLOCK_M; x += 4)
          mine4[x / 4] = make_float4(acc[x], acc[x + 1], acc[x + 2], acc[x + 3]);
        // the barrier orders the warpgroup's partial writes before one
        // thread's release-acquire arrival on the tile counter (cumulative
        // release); the second barrier passes the acquire on to all 128
        // threads, so no separate fences are needed
        named_bar_sync(1, 128);
        if (quarter == 0 && lane == 0) {
          const unsigned prev = atomic_add_acq_rel_gpu(p.counters + t, 1u);
          *last_flag = (prev == static_cast<unsigned>(ncontrib - 1));
        }
        named_bar_sync(1, 128);
        if (*last_flag) {
          // contributors in a fixed order (this CTA's own values from
          // registers); the loads of several contributors are in flight together
          float sum[BLOCK_M];
#pragma unroll
          for (int x = 0; x < BLOCK_M; ++x) sum[x] = 0.f;
#pragma unroll 4
          for (int q = 0; q < ncontrib; ++q) {
            const float4 *src = reinterpret_cast<const float4 *>(
                slot_base + static_cast<size_t>(q) * (DBLOCK_N * BLOCK_M) + r * BLOCK_M);
#pragma unroll
            for (int x = 0; x < BLOCK_M; x += 4) {
              float4 v4;
              if (q == idx)
                v4 = make_float4(acc[x], acc[x + 1], acc[x + 2], acc[x + 3]);
              else
                v4 = __ldcg(src + x / 4);
              sum[x] += v4.x;
              sum[x + 1] += v4.y;
              sum[x + 2] += v4.z;
              sum[x + 3] += v4.w;
            }
          }
#pragma unroll
          for (int x = 0; x < BLOCK_M; ++x)
            if (m0 + x < M) p.C[static_cast<size_t>(m0 + x) * N + n] = f32_to_16<BF16>(sum[x]);
          if (quarter == 0 && lane == 0) p.counters[t] = 0u;
        }
        named_bar_sync(1, 128);   // last_flag is reused by the next segment
      }
      if (quarter == 0 && lane == 0) TMW4_STAMP(11, jseg);
      pos.step(jend - jseg, S, NT);
      jseg = jend;
    }
  } else {
    // ------------------------------------------------------------ dequant
    const int dw = warp - DQ_WARP0;
    const int wg = dw >> 2;
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;            // weight column within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t slot0 = tmem + lane_addr + wg * WG_COLS + 2 * DCOLS;
    uint64_t *const my_tfull = tfull_bar + wg * TSW;
    uint64_t *const my_kfree = kfree_bar + wg * TSW;
    const int w_off = (r >> 6) * ATOM_BYTES + (r & 63) * 16;
    const int zshift = (r & 1) * 4;
    const bool has_zeros = p.zeros != nullptr;
    bool ok = true;
    unsigned c = 0;                               // this warpgroup's block counter
    UnitPos pos = pos0;
    pos.step(wg, S, NT);
    // reads block b of a stage: its two 16-byte words, scale and zero
    // shared-memory offsets of this thread's scale and zero byte for the
    // group of block b of a full stage (stages start on a multiple of 4
    // blocks, so the group index within the stage is b >> gshift)
    int sc_off[WKB], zp_off[WKB];
#pragma unroll
    for (int b = 0; b < WKB; ++b) {
      sc_off[b] = W_SC_OFF + ((b >> gshift) * DBLOCK_N + r) * 2;
      zp_off[b] = W_ZP_OFF + (b >> gshift) * (DBLOCK_N / 2) + (r >> 1);
    }
    auto read_scale_zero = [&](const uint8_t *st, int soff, int zoff, uint32_t &s2, uint32_t &zm2) {
      s2 = dup16(*reinterpret_cast<const uint16_t *>(st + soff));
      const uint32_t z =
          has_zeros ? (static_cast<uint32_t>(st[zoff]) >> zshift) & 0xFu : 8u;
      zm2 = zero_magic2<BF16>(z);
    };
    auto read_block = [&](const uint8_t *st, int b, int kbf, int gf, uint4 &v0, uint4 &v1,
                          uint32_t &s2, uint32_t &zm2) {
      const uint8_t *src = st + b * BLOCK_BYTES + w_off;
      v0 = *reinterpret_cast<const uint4 *>(src);
      v1 = *reinterpret_cast<const uint4 *>(src + 1024);
      const int gi = ((kbf + b) >> gshift) - gf;
      read_scale_zero(st, W_SC_OFF + (gi * DBLOCK_N + r) * 2, W_ZP_OFF + gi * (DBLOCK_N / 2) + (r >> 1),
                      s2, zm2);
    };
    // dequantizes one block into TMEM slot `slot` (stores not yet waited)
    auto put_block = [&](const uint4 &v0, const uint4 &v1, uint32_t s2, uint32_t zm2, unsigned slot) {
      uint32_t d0[16], d1[16];
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
      const uint32_t ta = slot0 + slot * DSLOT_COLS;
      tmem_st_16(ta, d0);
      tmem_st_16(ta + 16, d1);
    };
    // before writing block `cl`'s slot: the MMAs of block cl - TSW retired
    // (one thread issues the warpgroup's MMAs, so its commits complete in
    // order and this also covers every earlier block)
    auto slot_free = [&](unsigned cl, int step) -> bool {
      if (cl < static_cast<unsigned>(TSW)) return true;
      return mbar_wait_all(my_kfree + (cl & (TSW - 1)), ((cl / TSW) & 1u) ^ 1u, p.limit_ns,
                           abort_flag, p.err, SITE_DQ_AEMPTY, step, TMW4_SPIN(5));
    };
    // the weight stage `ws` is no longer needed by this warp: its data has
    // been dequantized and stored, and a generic-to-async proxy fence orders
    // the warp's shared-memory reads of it before the bulk copy that will
    // refill it; then arrive on the stage's empty barrier.  (Releasing the
    // stage as soon as its last block was in registers, without the fence,
    // let a refill corrupt a warp's weights now and then.)
    auto release_stage = [&](int ws_) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(wempty_bar + ws_);
    };
    // after the stores of blocks [c0, c0 + n): hand them to the MMA issuer
    auto publish = [&](unsigned c0, int n) {
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        for (int h = 0; h < n; ++h) mbar_arrive(my_tfull + ((c0 + h) & (TSW - 1)));
      }
    };
    for (int j = wg; j < nloc && ok; j += DQ_WG, pos.step(DQ_WG, S, NT)) {
      const int ws = j % WST;
      if (!mbar_wait_all(wfull_bar + ws, (j / WST) & 1, p.limit_ns, abort_flag, p.err, SITE_DQ_FULL,
                         j, TMW4_SPIN(4))) {
        ok = false;
        break;
      }
      const uint8_t *st = sW + ws * W_STAGE_BYTES;
      const int kbf = pos.s * WKB;
      const int nb = min(WKB, KB - kbf);
      const int gf = kbf >> gshift;
      if (nb == WKB) {
        // a full stage, two blocks at a time; the stage is released once its
        // last pair has been dequantized
#pragma unroll
        for (int pr = 0; pr < WKB / 2; ++pr) {
          uint4 v[2][2];
          uint32_t s2[2], zm2[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint8_t *src = st + (2 * pr + h) * BLOCK_BYTES + w_off;
            v[h][0] = *reinterpret_cast<const uint4 *>(src);
            v[h][1] = *reinterpret_cast<const uint4 *>(src + 1024);
            read_scale_zero(st, sc_off[2 * pr + h], zp_off[2 * pr + h], s2[h], zm2[h]);
          }
          if (!slot_free(c + 2 * pr + 1, j * WKB + 2 * pr)) {
            ok = false;
            break;
          }
          tc_fence_after();
          put_block(v[0][0], v[0][1], s2[0], zm2[0], (c + 2 * pr) & (TSW - 1));
          put_block(v[1][0], v[1][1], s2[1], zm2[1], (c + 2 * pr + 1) & (TSW - 1));
          publish(c + 2 * pr, 2);
          if (pr == WKB / 2 - 1) release_stage(ws);
        }
        if (wg == 0 && quarter == 2 && lane == 0) TMW4_STAMP(3, j * WKB);
        c += WKB;
      } else {
        // the ragged last stage of a tile: one block at a time
        for (int b = 0; b < nb; ++b) {
          uint4 v0, v1;
          uint32_t s2, zm2;
          read_block(st, b, kbf, gf, v0, v1, s2, zm2);
          if (!slot_free(c, j * WKB + b)) {
            ok = false;
            break;
          }
          tc_fence_after();
          put_block(v0, v1, s2, zm2, c & (TSW - 1));
          publish(c, 1);
          if (b == nb - 1) release_stage(ws);
          ++c;
        }
      }
    }
  }
#ifdef TMW4_TRACE
  // per-role finishing time of every CTA (slot by role, index 128 + CTA % 128)
  if (p.trace != nullptr && lane == 0) {
    const int role_slot = warp == 0 ? 6 : warp == 1 ? 10 : warp == ISSUE_WARP0 ? 12
                        : warp == EPI_WARP0 ? 11 : warp == DQ_WARP0 ? 7 : -1;
    if (role_slot >= 0)
      p.trace[role_slot * 256 + 128 + (blockIdx.x & 127)] = static_cast<long long>(globaltimer_ns());
  }
#endif
  // Lanes of the single-thread roles (producers, MMA issuer) leave their
  // branch at different times than the rest of their warp; reconverge
  // each warp first, because a CTA barrier counts a warp as arrived as soon
  // as any of its lanes reach it, and TMEM may only be freed once every
  // role, those lanes included, is done with it.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
#ifdef TMW4_TRACE
  if (threadIdx.x == 0 && p.trace != nullptr && blockIdx.x < 256)
    p.trace[14 * 256 + blockIdx.x] = static_cast<long long>(globaltimer_ns());
#endif
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
#ifdef TMW4_TRACE
    if (lane == 0 && p.trace != nullptr && blockIdx.x < 256)
      p.trace[5 * 256 + 128 + (blockIdx.x & 127)] = static_cast<long long>(globaltimer_ns());
#endif
    tmem_dealloc(tmem, TMEM_COLS);
#ifdef TMW4_TRACE
    if (lane == 0 && p.trace != nullptr && blockIdx.x < 256)
      p.trace[9 * 256 + blockIdx.x] = static_cast<long long>(globaltimer_ns());
#endif
  }
}

bool tc_decode_ok(int block_m, int dq_warps) {
  if (block_m != 16 && block_m != 32 && block_m != 64) return false;
  if (dq_warps != 4 && dq_warps != 8 && dq_warps != 12 && dq_warps != 16) return false;
  const int wg = dq_warps / 4;
  return dec_tsw(block_m, wg) >= 2 && dec_wst(block_m, wg) >= 2 * wg;
}

int tc_decode_slots(int block_m, int dq_warps) { return dec_tsw(block_m, dq_warps / 4); }

int tc_decode_kblocks_per_stage() { return WKB; }

void tc_decode_pipeline(int block_m, int dq_warps, int *weight_stages, int *act_stages_per_wg,
                        int *tmem_slots_per_wg) {
  const int wg = dq_warps / 4;
  *weight_stages = wg > 0 ? dec_wst(block_m, wg) : 0;
  *act_stages_per_wg = wg > 0 ? dec_asw(block_m, wg) : 0;
  *tmem_slots_per_wg = wg > 0 ? dec_tsw(block_m, wg) : 0;
}

void tc_decode_plan(int M, int N, int K, int block_m, int sms, int *grid, long long *tiles,
                    int *ws_slots) {
  const long long KB = K / DBLOCK_K;
  const long long S = (KB + WKB - 1) / WKB;
  const long long T = static_cast<long long>(N / DBLOCK_N) * ((M + block_m - 1) / block_m);
  const long long U = T * S;
  const long long G = std::max<long long>(1, std::min<long long>(sms, U));
  // contributors of a tile: the CTAs whose ranges meet its S units
  int maxc = 1;
  for (long long t = 0; t < T; ++t) {
    const int c = cta_of_unit((t + 1) * S - 1, U, G) - cta_of_unit(t * S, U, G) + 1;
    if (c > maxc) maxc = c;
  }
  *grid = static_cast<int>(G);
  *tiles = T;
  *ws_slots = maxc;
}

template <bool BF16, int BLOCK_M, int DQ_WG>
static cudaError_t launch_dec_t(const GemmArgs &a, const CUtensorMap &tmap, int grid, cudaStream_t st) {
  auto kern = tc_decode_kernel<BF16, BLOCK_M, DQ_WG>;
  const int smem = static_cast<int>(dec_smem_bytes(BLOCK_M, DQ_WG));
  cudaError_t e = smem_optin<tc_decode_kernel<BF16, BLOCK_M, DQ_WG>>(smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(dec_threads(DQ_WG)), static_cast<size_t>(smem), st,
                       a.pdl != 0, tmap, a);
}

template <bool BF16, int BLOCK_M>
static cudaError_t launch_dec_bm(const GemmArgs &a, const CUtensorMap &tmap, int dq, int grid,
                                 cudaStream_t st) {
  switch (dq) {
    case 4: return launch_dec_t<BF16, BLOCK_M, 1>(a, tmap, grid, st);
    case 8: return launch_dec_t<BF16, BLOCK_M, 2>(a, tmap, grid, st);
    case 12:
      if constexpr (dec_tsw(BLOCK_M, 3) >= 2) return launch_dec_t<BF16, BLOCK_M, 3>(a, tmap, grid, st);
      return cudaErrorInvalidValue;
    case 16:
      if constexpr (dec_tsw(BLOCK_M, 4) >= 2) return launch_dec_t<BF16, BLOCK_M, 4>(a, tmap, grid, st);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_tc_decode(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int block_m,
                             int dq_warps, int grid, cudaStream_t st) {
  switch (block_m) {
    case 16: return bf16 ? launch_dec_bm<true, 16>(a, tmap_a, dq_warps, grid, st)
                         : launch_dec_bm<false, 16>(a, tmap_a, dq_warps, grid, st);
    case 32: return bf16 ? launch_dec_bm<true, 32>(a, tmap_a, dq_warps, grid, st)
                         : launch_dec_bm<false, 32>(a, tmap_a, dq_warps, grid, st);
    case 64: return bf16 ? launch_dec_bm<true, 64>(a, tmap_a, dq_warps, grid, st)
                         : launch_dec_bm<false, 64>(a, tmap_a, dq_warps, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tmw4

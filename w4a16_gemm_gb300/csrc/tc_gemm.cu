// tc_gemm.cu -- W4A16 GEMM on the 5th-generation tensor cores (tcgen05).
//
// Blackwell restatement of the pages' parallel MMA-dequantization (TurboMind
// paper, pith.science review, Figure 9: tensor cores multiply tile k while
// the INT/FP ALUs dequantize tile k+1 and loads for later tiles are in
// flight).  The product is computed transposed, C^T = W^T A^T, so that the
// dequantized weight is the MMA's A operand and can live in tensor memory:
//
//   warp 0      TMA producer: one 2-D tensor load of the activation tile
//               (128-byte swizzle) plus 1-D bulk copies of the packed weight
//               tile (4 KB, contiguous in the packed layout), its scales and
//               zeros, into a ring of shared-memory stages (mbarrier
//               complete_tx).
//   warp 1      TMEM allocator and the single MMA-issuing thread:
//               tcgen05.mma kind::f16, D[128 x BLOCK_M] (fp32, TMEM) +=
//               A[128 x 16] (TMEM) * B[16 x BLOCK_M] (shared memory).
//   warps 2..   dequant warpgroups (stage i goes to warpgroup i % count); in
//               each, thread i owns weight column n0+i (TMEM lane i),
//               reads its 32-byte slice of the stage with two 128-bit shared
//               loads, dequantizes exactly (w = T(s*(q-z))) and writes the
//               32 packed pairs to a TMEM A stage with tcgen05.st; they then
//               run the epilogue (tcgen05.ld of D, convert, store C or the
//               split-K partial).
//
// Every mbarrier wait is bounded: a wait that gives up sets the device error
// word and a CTA-wide abort flag, every role leaves its loop, in-flight TMA
// copies and MMAs are waited for (again bounded) and TMEM is freed.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tc_epilogue.cuh"

namespace tmw4 {

namespace {

constexpr int BLOCK_N = 128;               // weight columns per CTA = MMA M
constexpr int BLOCK_K = 64;                // K per k-block (one TMEM A slot)
// bytes of one 64-K tile block and of one group row of zeros, for WB-bit codes
__host__ __device__ constexpr int w_kb_bytes(int wb) { return BLOCK_N * BLOCK_K * wb / 8; }   // 4096 / 8192
__host__ __device__ constexpr int zp_group_bytes(int wb) { return BLOCK_N * wb / 8; }          // 64 / 128
constexpr int SC_GROUP_BYTES = BLOCK_N * 2;           // 256: one group row of scales
constexpr int TMEM_A_COLS = BLOCK_K / 2;   // 32 columns of packed pairs per k-block

// k-blocks per shared-memory stage: small tiles move more weight per stage so
// that one stage (one bulk copy of contiguous tile blocks) amortises the
// fixed cost of issuing its copies.
__host__ __device__ constexpr int kbs_for(int block_m) {
  return block_m <= 16 ? 4 : block_m <= 64 ? 2 : 1;
}
__host__ __device__ constexpr int a_kb_bytes(int block_m) { return block_m * BLOCK_K * 2; }
__host__ __device__ constexpr int stage_bytes(int block_m, int wb = 4) {
  // (room for two groups per 64-K block: G = 32)
  return kbs_for(block_m) * (a_kb_bytes(block_m) + w_kb_bytes(wb) + 2 * SC_GROUP_BYTES + 2 * zp_group_bytes(wb));
}
// A copy takes ~1500 cycles to land under prefill load, so the ring must be
// deep enough to cover it: 256-row tiles take the six stages that fit.
__host__ __device__ constexpr int stages_for(int block_m, int wb = 4) {
  // (8-bit codes double the weight bytes of a stage: four stages at 256 rows)
  return block_m <= 64 ? 4 : block_m <= 128 ? 8 : wb == 4 ? 6 : 4;
}
// TMEM: D occupies columns [0, max(32, BLOCK_M)); the rest of a 256-column
// (BLOCK_M <= 128) or 512-column allocation is a ring of k-block A slots.
__host__ __device__ constexpr int tmem_a_col0(int block_m) { return block_m < 32 ? 32 : block_m; }
__host__ __device__ constexpr int tmem_cols(int block_m) { return block_m <= 128 ? 256 : 512; }
__host__ __device__ constexpr int tmem_a_stages(int block_m) {
  return (tmem_cols(block_m) - tmem_a_col0(block_m)) / TMEM_A_COLS;
}
// Every mbarrier wait here is a parity wait, which cannot tell phase c from
// phase c-2: it is correct only if, when a consumer starts waiting for the
// c-th completion of a barrier, completion c-1 is already known to have
// happened.  Copies issued in order may land out of order, so a dequant warp
// may rely only on completions it has observed itself.  With DQ_WG
// warpgroups taking alternate stages that holds iff
//   STAGES % DQ_WG == 0    (each shared-memory slot is always consumed by the
//                           same warpgroup, which saw the slot's previous fill)
//   TS >= (DQ_WG - 1) * KBS + 1
//                          (a warp's previous wait on a TMEM slot proves the
//                           MMAs two uses back retired; MMAs retire in order)
// A randomized model of this protocol (tests/test_pipeline_protocol.py)
// checks both conditions.
__host__ __device__ constexpr bool variant_ok(int block_m, int dq_wg, int wb = 4) {
  return stages_for(block_m, wb) % dq_wg == 0 &&
         tmem_a_stages(block_m) >= (dq_wg - 1) * kbs_for(block_m) + 1;
}
__host__ __device__ constexpr size_t smem_bytes_for(int block_m, int wb = 4) {
  return 1024 /* alignment slack */ +
         static_cast<size_t>(stages_for(block_m, wb)) * stage_bytes(block_m, wb) +
         512 /* barriers and flags */;
}

}  // namespace


// DQ_WG dequant warpgroups; warpgroup g dequantizes the shared-memory stages
// j with j % DQ_WG == g, so DQ_WG stages are in flight in the ALUs at once.
// WB: bits per weight code, 4, or 8 (int8 with byte zeros, or FP8 E4M3 codes,
// GemmArgs::fp8); an 8-bit tile block is 16-byte chunks of 16 consecutive K
// of one column, chunk kq * 128 + c.
template <bool BF16, int BLOCK_M, int DQ_WG, int WB>
__global__ void __launch_bounds__(64 + 128 * DQ_WG, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs p) {
  constexpr int STAGES = stages_for(BLOCK_M, WB);
  constexpr int W_KB_BYTES = w_kb_bytes(WB);
  constexpr int ZP_GROUP_BYTES = zp_group_bytes(WB);
  constexpr int KBS = kbs_for(BLOCK_M);
  constexpr int A_KB = a_kb_bytes(BLOCK_M);
  constexpr int A_STAGE = KBS * A_KB;
  constexpr int W_STAGE = KBS * W_KB_BYTES;
  constexpr int SC_STAGE = 2 * KBS * SC_GROUP_BYTES;   // room for 2 KBS groups (G = 32)
  constexpr int ZP_STAGE = 2 * KBS * ZP_GROUP_BYTES;
  constexpr int TMEM_COLS = tmem_cols(BLOCK_M);
  constexpr int A_COL0 = tmem_a_col0(BLOCK_M);
  constexpr int TS = tmem_a_stages(BLOCK_M);
  constexpr uint32_t IDESC = idesc_f16(BF16 ? 1u : 0u, 128u, static_cast<uint32_t>(BLOCK_M));
  static_assert(BLOCK_M % 16 == 0 && BLOCK_M >= 16 && BLOCK_M <= 256, "MMA N");
  static_assert(DQ_WG == 1 || DQ_WG == 2 || DQ_WG == 4, "dequant warpgroups");
  static_assert(TS >= 2, "TMEM A slots");
  static_assert(variant_ok(BLOCK_M, DQ_WG, WB), "parity waits need at most one phase of lead");
  static_assert(WB == 4 || WB == 8, "code width");
  static_assert(A_KB % 1024 == 0, "swizzle atoms");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align_smem_1024(smem_raw);
  uint8_t *sA = smem;                              // [STAGES][KBS][BLOCK_M x 128 B]
  uint8_t *sW = sA + STAGES * A_STAGE;             // [STAGES][KBS][4096]
  uint8_t *sSC = sW + STAGES * W_STAGE;            // [STAGES][groups][256]
  uint8_t *sZP = sSC + STAGES * SC_STAGE;          // [STAGES][groups][64]
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(sZP + STAGES * ZP_STAGE);
  uint64_t *empty_bar = full_bar + STAGES;
  uint64_t *afull_bar = empty_bar + STAGES;
  uint64_t *aempty_bar = afull_bar + TS;
  uint64_t *accum_bar = aempty_bar + TS;
  uint64_t *drain_bar = accum_bar + 1;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain_bar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  int *last_flag = reinterpret_cast<int *>(tmem_holder + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x;
  const int n0 = nt * BLOCK_N;
  const int m0 = blockIdx.y * BLOCK_M;
  const int split = blockIdx.z;
  const int KB = p.K / BLOCK_K;
  const int G_rows = p.K / p.group;
  const int kb0 = split * p.kb_per_split;
  const int nkb = max(0, min(KB, kb0 + p.kb_per_split) - kb0);
  const int nstages = (nkb + KBS - 1) / KBS;

  if (threadIdx.x == 0) {
    TMW4_STAMP(7, 1);
    *abort_flag = 0;
    *last_flag = 0;
    prefetch_tensormap(&tmap_a);
  }
  {
    // one barrier per thread; the barriers are contiguous, in the order
    // full, empty, afull, aempty, accum, drain
    constexpr int NBAR = 2 * STAGES + 2 * TS + 2;
    static_assert(NBAR <= 64 + 128 * DQ_WG, "one thread per barrier");
    const int b = threadIdx.x;
    if (b < NBAR) {
      int cnt = 1;
      if (b >= STAGES && b < 2 * STAGES) cnt = 1 + 4;   // MMA commit + the 4 warps of one warpgroup
      if (b >= 2 * STAGES && b < 2 * STAGES + TS) cnt = 4;
      mbar_init(full_bar + b, cnt);
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
  // the prologue above overlaps the previous kernel in the stream; nothing
  // below runs before it has completed
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nstages; ++j) {
        const int s = j % STAGES;
        const uint32_t ph = (j / STAGES) & 1;
        if (j >= STAGES &&
            !mbar_wait_idle(empty_bar + s, ph ^ 1u, p.limit_ns, abort_flag, p.err, SITE_PRODUCER_EMPTY, j))
          break;
        const int kbf = kb0 + j * KBS;
        const int nb = min(KBS, nkb - j * KBS);
        const int gf = (kbf * BLOCK_K) / p.group;
        const int gl = ((kbf + nb) * BLOCK_K - 1) / p.group;
        const int ng = gl - gf + 1;
        const uint32_t a_bytes = (p.act_map_3d ? KBS : nb) * A_KB;
        const uint32_t tx = a_bytes + nb * W_KB_BYTES + ng * SC_GROUP_BYTES +
                            (p.zeros != nullptr ? ng * ZP_GROUP_BYTES : 0);
        mbar_arrive_expect_tx(full_bar + s, tx);
        if (p.act_map_3d) {
          tma_load_3d(sA + s * A_STAGE, &tmap_a, 0, m0, kbf, full_bar + s);
        } else {
          for (int b = 0; b < nb; ++b)
            tma_load_2d(sA + s * A_STAGE + b * A_KB, &tmap_a, (kbf + b) * BLOCK_K, m0, full_bar + s);
        }
        tma_bulk_g2s(sW + s * W_STAGE, p.qw + (static_cast<size_t>(nt) * KB + kbf) * W_KB_BYTES,
                     nb * W_KB_BYTES, full_bar + s);
        tma_bulk_g2s(sSC + s * SC_STAGE, p.scales + (static_cast<size_t>(nt) * G_rows + gf) * BLOCK_N,
                     ng * SC_GROUP_BYTES, full_bar + s);
        if (p.zeros != nullptr)
          tma_bulk_g2s(sZP + s * ZP_STAGE,
                       p.zeros + (static_cast<size_t>(nt) * G_rows + gf) * ZP_GROUP_BYTES,
                       ng * ZP_GROUP_BYTES, full_bar + s);
        TMW4_STAMP(0, j);
        issued = j + 1;
      }
      // drain: every copy issued must have landed before the CTA exits
      for (int s = 0; s < STAGES && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / STAGES) * STAGES;
        mbar_wait_bounded(full_bar + s, (last / STAGES) & 1, p.limit_ns, nullptr, p.err, SITE_DRAIN_TMA, last);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      bool any = false, ok = true;
      // descriptor of the B tile (activations) of stage 0, block 0; other
      // tiles are a constant number of 16-byte units further on
      const uint64_t desc0 = smem_desc_k128(smem_u32(sA));
      uint32_t a_slot = tmem + A_COL0;      // TMEM A slot of block i (ring of TS)
      int t = 0;
      for (int j = 0; j < nstages && ok; ++j) {
        const int s = j % STAGES;
        if (!mbar_wait_bounded(full_bar + s, (j / STAGES) & 1, p.limit_ns, abort_flag, p.err, SITE_MMA_FULL, j)) {
          ok = false;
          break;
        }
        const int nb = min(KBS, nkb - j * KBS);
        const uint64_t desc_s = desc0 + static_cast<uint64_t>((s * A_STAGE) >> 4);
        for (int b = 0; b < nb; ++b) {
          const int i = j * KBS + b;
#ifdef TMW4_TRACE
          TMW4_STAMP(7, 2 + i);
#endif
          if (!mbar_wait_bounded(afull_bar + t, (i / TS) & 1, p.limit_ns, abort_flag, p.err, SITE_MMA_AFULL, i)) {
            ok = false;
            break;
          }
          TMW4_STAMP(4, i);
          tc_fence_after();
          tc_mma_ts_kblock(tmem, a_slot, desc_s + static_cast<uint64_t>((b * A_KB) >> 4), IDESC,
                           i == 0 ? 1u : 0u);
          tc_commit(aempty_bar + t);
          TMW4_STAMP(5, i);
          any = true;
          if (++t == TS) {
            t = 0;
            a_slot = tmem + A_COL0;
          } else {
            a_slot += TMEM_A_COLS;
          }
        }
        if (ok) tc_commit(empty_bar + s);
      }
      if (ok && any) {
        tc_commit(accum_bar);
      } else if (any) {
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, p.limit_ns, nullptr, p.err, SITE_DRAIN_MMA, 0);
      }
    }
  } else {
    // ------------------------------------------------- dequant + epilogue
    const int dw = warp - 2;
    const int wg = dw >> 2;                   // this warp's warpgroup
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;        // weight column within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int atom = r >> 6, nl = r & 63;
    // this thread's codes in a stage: 4-bit, two chunks (K 0-31, 32-63) of
    // its column in its atom; 8-bit, four chunks 2048 bytes apart
    const uint8_t *wsrc = WB == 4 ? sW + atom * ATOM_BYTES + nl * 16 : sW + r * 16;
    bool ok = true;
    for (int j = wg; j < nstages && ok; j += DQ_WG) {
      const int s = j % STAGES;
      // the warp agrees on the outcome, so tcgen05.st below is always executed
      // by the whole warp
      if (!mbar_wait_warp(full_bar + s, (j / STAGES) & 1, p.limit_ns, abort_flag, p.err,
                          SITE_DQ_FULL, j)) {
        ok = false;
        break;
      }
      if (quarter == 2 && lane == 0) TMW4_STAMP(1, j);
      const int kbf = kb0 + j * KBS;
      const int nb = min(KBS, nkb - j * KBS);
      const int gf = (kbf * BLOCK_K) / p.group;
      for (int b = 0; b < nb; ++b) {
        const int i = j * KBS + b;
        const int t = i % TS;
        if (i >= TS && !mbar_wait_warp(aempty_bar + t, ((i / TS) & 1) ^ 1u, p.limit_ns,
                                       abort_flag, p.err, SITE_DQ_AEMPTY, i)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (quarter == 2 && lane == 0) TMW4_STAMP(2, i);
        const int gi = ((kbf + b) * BLOCK_K) / p.group - gf;
        uint32_t d0[16], d1[16];
        if constexpr (WB == 8) {
          // 8-bit: scales and byte zeros of the block's two 32-K halves
          const uint8_t *src = wsrc + s * W_STAGE + b * W_KB_BYTES;
          uint4 v[4];
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) v[kq] = *reinterpret_cast<const uint4 *>(src + kq * 2048);
          if (b == nb - 1) {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar + s);   // last read of this stage done
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int gh = p.group == 32 ? gi + h : gi;
            const uint16_t sc = reinterpret_cast<const uint16_t *>(sSC + s * SC_STAGE + gh * SC_GROUP_BYTES)[r];
            const uint32_t z = p.zeros != nullptr ? sZP[s * ZP_STAGE + gh * ZP_GROUP_BYTES + r] : 128u;
            const uint32_t s2 = dup16(sc), zm2 = zero_magic2<false>(z);
            const float sf = BF16 ? __uint_as_float(static_cast<uint32_t>(sc) << 16) : __half2float(__ushort_as_half(sc));
            uint32_t *d = h == 0 ? d0 : d1;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint4 vv = v[2 * h + kk];
              const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t o[2];
                dequant_word8<BF16>(w[j], p.fp8 != 0, zm2, z, s2, sf, o);
                d[8 * kk + 2 * j] = o[0];
                d[8 * kk + 2 * j + 1] = o[1];
              }
            }
          }
        } else {
          const uint16_t sc =
              reinterpret_cast<const uint16_t *>(sSC + s * SC_STAGE + gi * SC_GROUP_BYTES)[r];
          const uint32_t z =
              p.zeros != nullptr
                  ? (static_cast<uint32_t>(sZP[s * ZP_STAGE + gi * ZP_GROUP_BYTES + (r >> 1)]) >>
                     ((r & 1) * 4)) & 0xFu
                  : 8u;
          const uint8_t *src = wsrc + s * W_STAGE + b * W_KB_BYTES;
          const uint4 v0 = *reinterpret_cast<const uint4 *>(src);
          const uint4 v1 = *reinterpret_cast<const uint4 *>(src + 1024);
#ifdef TMW4_TRACE
          if (p.trace != nullptr && quarter == 2 && lane == 0 && ((v0.x ^ v1.y) == 0x9E3779B9u)) p.trace[8 * 256] = 1;
          if (quarter == 2 && lane == 0) TMW4_STAMP(8, i);
#endif
          if (b == nb - 1) {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar + s);   // last read of this stage done
          }
          const uint32_t s2 = dup16(sc), zm2 = zero_magic2<BF16>(z);
          // the block's second 32-K half has a group of its own only when G = 32
          uint32_t s2b = s2, zm2b = zm2;
          if (p.group == 32) {
            const uint16_t sc1 =
                reinterpret_cast<const uint16_t *>(sSC + s * SC_STAGE + (gi + 1) * SC_GROUP_BYTES)[r];
            const uint32_t z1 =
                p.zeros != nullptr
                    ? (static_cast<uint32_t>(sZP[s * ZP_STAGE + (gi + 1) * ZP_GROUP_BYTES + (r >> 1)]) >>
                       ((r & 1) * 4)) & 0xFu
                    : 8u;
            s2b = dup16(sc1);
            zm2b = zero_magic2<BF16>(z1);
          }
          {
            const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
            const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t o[4];
              dequant_word<BF16>(w0[q4], zm2, s2, o);
#pragma unroll
              for (int q = 0; q < 4; ++q) d0[4 * q4 + q] = o[q];
              dequant_word<BF16>(w1[q4], zm2b, s2b, o);
#pragma unroll
              for (int q = 0; q < 4; ++q) d1[4 * q4 + q] = o[q];
            }
          }
        }
#ifdef TMW4_TRACE
        if (p.trace != nullptr && quarter == 2 && lane == 0 && ((d0[3] ^ d1[7]) == 0x9E3779B9u)) p.trace[8 * 256 + 1] = 1;
        if (quarter == 2 && lane == 0) TMW4_STAMP(9, i);
#endif
        __syncwarp();
        const uint32_t ta = tmem + lane_addr + A_COL0 + t * TMEM_A_COLS;
        tmem_st_16(ta, d0);
        tmem_st_16(ta + 16, d1);
#ifdef TMW4_TRACE
        if (quarter == 2 && lane == 0) TMW4_STAMP(10, i);
#endif
        tmem_wait_st();
#ifdef TMW4_TRACE
        if (quarter == 2 && lane == 0) TMW4_STAMP(11, i);
#endif
        tc_fence_before();
        __syncwarp();
        if (quarter == 2 && lane == 0) TMW4_STAMP(3, i);
#ifdef TMW4_TRACE
        if (lane == 0) TMW4_STAMP(12 + quarter, i);
#endif
        if (lane == 0) mbar_arrive(afull_bar + t);
      }
    }

    // ------------------------------------------------------------ epilogue
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (ok && nkb > 0)
      ok = mbar_wait_warp(accum_bar, 0, p.limit_ns, abort_flag, p.err, SITE_EPI_ACCUM, 0);
    if (dw == 0 && lane == 0) TMW4_STAMP(6, 0);
    tc_fence_after();
    // the stage ring is idle once every MMA has retired: reuse it to stage C
    tc_epilogue<BF16, BLOCK_M, DQ_WG>(p, tmem + lane_addr, wg, dw, lane, r, n0, m0, split, ok,
                                      nkb > 0 ? 1 : 0, 0u, last_flag, smem);
  }

  // Lanes of the single-thread roles (producers, MMA issuer) leave their
  // branch at different times than the rest of their warp; reconverge
  // each warp first, because a CTA barrier counts a warp as arrived as soon
  // as any of its lanes reach it, and TMEM may only be freed once every
  // role, those lanes included, is done with it.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) TMW4_STAMP(6, 1);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

size_t tc_smem_bytes(int block_m) { return smem_bytes_for(block_m); }
int tc_stages(int block_m) { return stages_for(block_m); }
int tc_kblocks_per_stage(int block_m) { return kbs_for(block_m); }
void tc_pipeline(int block_m, int *stages, int *kbs, int *tmem_slots) {
  *stages = stages_for(block_m);
  *kbs = kbs_for(block_m);
  *tmem_slots = tmem_a_stages(block_m);
}
bool tc_variant_ok(int block_m, int dq_warps, int wbits) {
  return (dq_warps == 4 || dq_warps == 8 || dq_warps == 16) &&
         (wbits == 8 ? variant_ok(block_m, dq_warps / 4, 8) : variant_ok(block_m, dq_warps / 4, 4));
}

template <bool BF16, int BLOCK_M, int DQ_WG, int WB>
static cudaError_t launch_tc_t(const GemmArgs &a, const CUtensorMap &tmap, cudaStream_t st) {
  auto kern = tc_gemm_kernel<BF16, BLOCK_M, DQ_WG, WB>;
  const size_t smem = smem_bytes_for(BLOCK_M, WB);
  cudaError_t e = smem_optin<tc_gemm_kernel<BF16, BLOCK_M, DQ_WG, WB>>(static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.N / BLOCK_N, (a.M + BLOCK_M - 1) / BLOCK_M, a.splits);
  return launch_kernel(kern, grid, dim3(64 + 128 * DQ_WG), smem, st, a.pdl != 0, tmap, a);
}

template <bool BF16, int BLOCK_M, int WB>
static cudaError_t launch_tc_bm(const GemmArgs &a, const CUtensorMap &tmap, int dq_warps,
                                cudaStream_t st) {
  switch (dq_warps) {
    case 4: return launch_tc_t<BF16, BLOCK_M, 1, WB>(a, tmap, st);
    case 8:
      if constexpr (variant_ok(BLOCK_M, 2, WB)) return launch_tc_t<BF16, BLOCK_M, 2, WB>(a, tmap, st);
      return cudaErrorInvalidValue;
    case 16:
      if constexpr (variant_ok(BLOCK_M, 4, WB)) return launch_tc_t<BF16, BLOCK_M, 4, WB>(a, tmap, st);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <bool BF16, int WB>
static cudaError_t launch_tc_dtype(const GemmArgs &a, const CUtensorMap &tmap, int block_m,
                                   int dq, cudaStream_t st) {
  switch (block_m) {
    case 16: return launch_tc_bm<BF16, 16, WB>(a, tmap, dq, st);
    case 32: return launch_tc_bm<BF16, 32, WB>(a, tmap, dq, st);
    case 64: return launch_tc_bm<BF16, 64, WB>(a, tmap, dq, st);
    case 128: return launch_tc_bm<BF16, 128, WB>(a, tmap, dq, st);
    case 256: return launch_tc_bm<BF16, 256, WB>(a, tmap, dq, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_tc(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int block_m,
                      int dq_warps, cudaStream_t st) {
  if (a.wbits == 8)
    return bf16 ? launch_tc_dtype<true, 8>(a, tmap_a, block_m, dq_warps, st)
                : launch_tc_dtype<false, 8>(a, tmap_a, block_m, dq_warps, st);
  return bf16 ? launch_tc_dtype<true, 4>(a, tmap_a, block_m, dq_warps, st)
              : launch_tc_dtype<false, 4>(a, tmap_a, block_m, dq_warps, st);
}

// ------------------------------------------------------ bounded-wait self test
__global__ void wait_selftest_kernel(unsigned int *err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives on `bar`: the wait must give up after limit_ns
    mbar_wait_bounded(&bar, 0, limit_ns, &abort_flag, err, SITE_SELFTEST, 0);
  }
  __syncwarp();
  __syncthreads();
}

cudaError_t launch_wait_selftest(unsigned int *err, unsigned long long limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace tmw4

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
//   warps 2..   dequant warps: thread i owns weight column n0+i (TMEM lane i),
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

namespace tmw4 {

namespace {

constexpr int BLOCK_N = 128;               // weight columns per CTA = MMA M
constexpr int BLOCK_K = 64;                // K per stage = one atom row
constexpr int W_STAGE_BYTES = BLOCK_N * BLOCK_K / 2;  // 4096
constexpr int SC_STAGE_BYTES = BLOCK_N * 2;            // 256
constexpr int ZP_STAGE_BYTES = BLOCK_N / 2;            // 64
constexpr int TMEM_A_STAGES = 4;
constexpr int TMEM_A_COLS = BLOCK_K / 2;   // 32 columns of packed pairs per stage

__host__ __device__ constexpr int stages_for(int block_m) {
  return block_m <= 16 ? 16 : block_m <= 32 ? 12 : block_m <= 64 ? 8 : block_m <= 128 ? 8 : 5;
}
__host__ __device__ constexpr int a_stage_bytes(int block_m) { return block_m * BLOCK_K * 2; }
__host__ __device__ constexpr int tmem_a_col0(int block_m) { return block_m < 32 ? 32 : block_m; }
__host__ __device__ constexpr int tmem_cols(int block_m) {
  // power of two >= D columns + A stages
  return (tmem_a_col0(block_m) + TMEM_A_STAGES * TMEM_A_COLS) <= 128   ? 128
         : (tmem_a_col0(block_m) + TMEM_A_STAGES * TMEM_A_COLS) <= 256 ? 256
                                                                       : 512;
}
__host__ __device__ constexpr size_t smem_bytes_for(int block_m) {
  return 1024 /* alignment slack */ +
         static_cast<size_t>(stages_for(block_m)) *
             (a_stage_bytes(block_m) + W_STAGE_BYTES + SC_STAGE_BYTES + ZP_STAGE_BYTES) +
         512 /* barriers and flags */;
}

template <bool BF16>
__device__ __forceinline__ uint16_t f32_to_16(float x) {
  if constexpr (BF16) {
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&b);
  } else {
    __half h = __float2half_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace

template <bool BF16, int BLOCK_M, int DQ_WARPS>
__global__ void __launch_bounds__(64 + 32 * DQ_WARPS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs p) {
  constexpr int STAGES = stages_for(BLOCK_M);
  constexpr int A_BYTES = a_stage_bytes(BLOCK_M);
  constexpr int TMEM_COLS = tmem_cols(BLOCK_M);
  constexpr int A_COL0 = tmem_a_col0(BLOCK_M);
  constexpr uint32_t IDESC = idesc_f16(BF16 ? 1u : 0u, 128u, static_cast<uint32_t>(BLOCK_M));
  constexpr int DQ_THREADS = 32 * DQ_WARPS;
  constexpr int PARTS = DQ_WARPS / 4;       // dequant warps per TMEM lane quarter
  constexpr int HALVES_PER_PART = 2 / PARTS;
  static_assert(BLOCK_M % 16 == 0 && BLOCK_M >= 16 && BLOCK_M <= 256, "MMA N");
  static_assert(DQ_WARPS == 4 || DQ_WARPS == 8, "dequant warps");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;                                         // [STAGES][A_BYTES]
  uint8_t *sW = sA + STAGES * A_BYTES;                        // [STAGES][4096]
  uint8_t *sSC = sW + STAGES * W_STAGE_BYTES;                 // [STAGES][256]
  uint8_t *sZP = sSC + STAGES * SC_STAGE_BYTES;               // [STAGES][64]
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(sZP + STAGES * ZP_STAGE_BYTES);
  uint64_t *empty_bar = full_bar + STAGES;
  uint64_t *afull_bar = empty_bar + STAGES;
  uint64_t *aempty_bar = afull_bar + TMEM_A_STAGES;
  uint64_t *accum_bar = aempty_bar + TMEM_A_STAGES;
  uint64_t *drain_bar = accum_bar + 1;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain_bar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  int *last_flag = reinterpret_cast<int *>(tmem_holder + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BLOCK_N;
  const int m0 = blockIdx.y * BLOCK_M;
  const int split = blockIdx.z;
  const int KB = p.K / BLOCK_K;
  const int kb0 = split * p.kb_per_split;
  const int nkb = max(0, min(KB, kb0 + p.kb_per_split) - kb0);
  const int N = p.N, M = p.M;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar + s, 1);
      mbar_init(empty_bar + s, 1 + DQ_WARPS);
    }
    for (int t = 0; t < TMEM_A_STAGES; ++t) {
      mbar_init(afull_bar + t, DQ_WARPS);
      mbar_init(aempty_bar + t, 1);
    }
    mbar_init(accum_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmap_a);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t tx = A_BYTES + W_STAGE_BYTES + SC_STAGE_BYTES +
                          (p.zeros != nullptr ? ZP_STAGE_BYTES : 0);
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (i >= STAGES &&
            !mbar_wait_bounded(empty_bar + s, ph ^ 1u, p.limit_ns, abort_flag, p.err))
          break;
        const int kb = kb0 + i;
        const int g = (kb * BLOCK_K) / p.group;
        mbar_arrive_expect_tx(full_bar + s, tx);
        tma_load_2d(sA + s * A_BYTES, &tmap_a, kb * BLOCK_K, m0, full_bar + s);
        tma_bulk_g2s(sW + s * W_STAGE_BYTES,
                     p.qw + (static_cast<size_t>(kb) * (N / ATOM_N) + n0 / ATOM_N) * ATOM_BYTES,
                     W_STAGE_BYTES, full_bar + s);
        tma_bulk_g2s(sSC + s * SC_STAGE_BYTES, p.scales + static_cast<size_t>(g) * N + n0,
                     SC_STAGE_BYTES, full_bar + s);
        if (p.zeros != nullptr)
          tma_bulk_g2s(sZP + s * ZP_STAGE_BYTES, p.zeros + static_cast<size_t>(g) * (N / 2) + n0 / 2,
                       ZP_STAGE_BYTES, full_bar + s);
        issued = i + 1;
      }
      // drain: every copy issued must have landed before the CTA exits
      for (int s = 0; s < STAGES && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / STAGES) * STAGES;
        mbar_wait_bounded(full_bar + s, (last / STAGES) & 1, p.limit_ns, nullptr, p.err);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      bool any = false, ok = true;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const int t = i % TMEM_A_STAGES;
        if (!mbar_wait_bounded(full_bar + s, (i / STAGES) & 1, p.limit_ns, abort_flag, p.err) ||
            !mbar_wait_bounded(afull_bar + t, (i / TMEM_A_STAGES) & 1, p.limit_ns, abort_flag,
                               p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(sA + s * A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BLOCK_K / 16; ++kk) {
          tc_mma_ts(tmem, tmem + A_COL0 + t * TMEM_A_COLS + kk * 8,
                    smem_desc_k128(a_base + kk * 32), IDESC, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(empty_bar + s);
        tc_commit(aempty_bar + t);
        any = true;
      }
      if (ok && any) {
        tc_commit(accum_bar);
      } else if (any) {
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, p.limit_ns, nullptr, p.err);
      }
    }
  } else {
    // ------------------------------------------------- dequant + epilogue
    const int dw = warp - 2;
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int part = dw / 4;                  // which K half(s) of the stage
    const int r = quarter * 32 + lane;        // weight column within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int atom = r >> 6, nl = r & 63;
    bool ok = true;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      const int t = i % TMEM_A_STAGES;
      // every lane waits (acquire for its own loads); the warp then agrees,
      // so tcgen05.st below is always executed by the whole warp
      bool got = mbar_wait_bounded(full_bar + s, (i / STAGES) & 1, p.limit_ns, abort_flag, p.err);
      if (got && i >= TMEM_A_STAGES)
        got = mbar_wait_bounded(aempty_bar + t, ((i / TMEM_A_STAGES) & 1) ^ 1u, p.limit_ns,
                                abort_flag, p.err);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint16_t sc = reinterpret_cast<const uint16_t *>(sSC + s * SC_STAGE_BYTES)[r];
      const uint32_t z = p.zeros != nullptr
                             ? (static_cast<uint32_t>(sZP[s * ZP_STAGE_BYTES + (r >> 1)]) >>
                                ((r & 1) * 4)) & 0xFu
                             : 8u;
      uint4 v[HALVES_PER_PART];
#pragma unroll
      for (int hh = 0; hh < HALVES_PER_PART; ++hh) {
        const int h = part * HALVES_PER_PART + hh;
        v[hh] = *reinterpret_cast<const uint4 *>(sW + s * W_STAGE_BYTES + atom * ATOM_BYTES +
                                                 h * 1024 + nl * 16);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar + s);
      const uint32_t s2 = dup16(sc), zm2 = zero_magic2<BF16>(z);
      __syncwarp();
#pragma unroll
      for (int hh = 0; hh < HALVES_PER_PART; ++hh) {
        const int h = part * HALVES_PER_PART + hh;
        uint32_t d[16];
        const uint32_t w[4] = {v[hh].x, v[hh].y, v[hh].z, v[hh].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t o[4];
          dequant_word<BF16>(w[j], zm2, s2, o);
#pragma unroll
          for (int q = 0; q < 4; ++q) d[4 * j + q] = o[q];
        }
        tmem_st_16(tmem + lane_addr + A_COL0 + t * TMEM_A_COLS + h * 16, d);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(afull_bar + t);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && nkb > 0) ok = mbar_wait_bounded(accum_bar, 0, p.limit_ns, abort_flag, p.err);
    ok = __all_sync(0xFFFFFFFFu, ok);
    tc_fence_after();
    const int n = n0 + r;
    const bool direct = (p.splits == 1);
    if (ok) {
      // columns of D are rows m of C; each part takes alternate 16-column chunks
      for (int c0 = part * 16; c0 < BLOCK_M; c0 += 16 * PARTS) {
        if (m0 + c0 >= M) break;  // warp-uniform
        uint32_t v[16];
        __syncwarp();
        if (nkb > 0) {
          tmem_ld_16(tmem + lane_addr + c0, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = m0 + c0 + j;
          if (m < M) {
            const float x = __uint_as_float(v[j]);
            if (direct)
              p.C[static_cast<size_t>(m) * N + n] = f32_to_16<BF16>(x);
            else
              p.ws[(static_cast<size_t>(split) * M + m) * N + n] = x;
          }
        }
      }
    }
    if (!direct) {
      __threadfence();
      named_bar_sync(1, DQ_THREADS);
      unsigned int *ctr = p.counters + (static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x);
      if (dw == 0 && lane == 0) {
        const unsigned prev = atomicAdd(ctr, 1u);
        *last_flag = (prev == static_cast<unsigned>(p.splits - 1));
      }
      named_bar_sync(1, DQ_THREADS);
      if (*last_flag) {
        __threadfence();
        for (int c0 = part; c0 < BLOCK_M; c0 += PARTS) {
          const int m = m0 + c0;
          if (m >= M) break;
          float acc = 0.f;
          for (int s = 0; s < p.splits; ++s)
            acc += __ldcg(p.ws + (static_cast<size_t>(s) * M + m) * N + n);
          p.C[static_cast<size_t>(m) * N + n] = f32_to_16<BF16>(acc);
        }
        if (dw == 0 && lane == 0) *ctr = 0u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

size_t tc_smem_bytes(int block_m) { return smem_bytes_for(block_m); }
int tc_stages(int block_m) { return stages_for(block_m); }

template <bool BF16, int BLOCK_M, int DQ_WARPS>
static cudaError_t launch_tc_t(const GemmArgs &a, const CUtensorMap &tmap, cudaStream_t st) {
  auto kern = tc_gemm_kernel<BF16, BLOCK_M, DQ_WARPS>;
  const size_t smem = smem_bytes_for(BLOCK_M);
  static int attr_device = -1;  // shared-memory opt-in, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_device != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_device = dev;
  }
  dim3 grid(a.N / BLOCK_N, (a.M + BLOCK_M - 1) / BLOCK_M, a.splits);
  kern<<<grid, 64 + 32 * DQ_WARPS, smem, st>>>(tmap, a);
  return cudaGetLastError();
}

template <bool BF16>
static cudaError_t launch_tc_dtype(const GemmArgs &a, const CUtensorMap &tmap, int block_m,
                                   int dq, cudaStream_t st) {
  if (dq == 4) {
    switch (block_m) {
      case 16: return launch_tc_t<BF16, 16, 4>(a, tmap, st);
      case 32: return launch_tc_t<BF16, 32, 4>(a, tmap, st);
      case 64: return launch_tc_t<BF16, 64, 4>(a, tmap, st);
      case 128: return launch_tc_t<BF16, 128, 4>(a, tmap, st);
      case 256: return launch_tc_t<BF16, 256, 4>(a, tmap, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (dq == 8) {
    switch (block_m) {
      case 16: return launch_tc_t<BF16, 16, 8>(a, tmap, st);
      case 32: return launch_tc_t<BF16, 32, 8>(a, tmap, st);
      case 64: return launch_tc_t<BF16, 64, 8>(a, tmap, st);
      case 128: return launch_tc_t<BF16, 128, 8>(a, tmap, st);
      case 256: return launch_tc_t<BF16, 256, 8>(a, tmap, st);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_tc(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int block_m,
                      int dq_warps, cudaStream_t st) {
  return bf16 ? launch_tc_dtype<true>(a, tmap_a, block_m, dq_warps, st)
              : launch_tc_dtype<false>(a, tmap_a, block_m, dq_warps, st);
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
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives on `bar`: the wait must give up after limit_ns
    mbar_wait_bounded(&bar, 0, limit_ns, &abort_flag, err);
  }
  __syncthreads();
}

cudaError_t launch_wait_selftest(unsigned int *err, unsigned long long limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace tmw4

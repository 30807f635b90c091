// tc_epilogue.cuh -- the output stage shared by the tcgen05 kernels: read the
// fp32 accumulator from TMEM, round once to the 16-bit output type, or write
// split-K partials and let the last CTA of the tile sum them in split order.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace tmw4 {

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

// bar.sync counts a whole warp as arrived as soon as any of its threads
// executes it.  A thread still inside a lane-0 branch (the counter atomic
// just before the fix-up barriers) would then miss the barrier and arrive at
// the next one instead, so every warp reconverges first.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Called by all DQ_WG * 128 epilogue threads of the CTA.  Thread (wg, lane
// quarter, lane) owns weight column n = n0 + r with r = 32 * quarter + lane
// (TMEM lane r); D's columns are the rows m0.. of C.  The result is the sum,
// in a fixed order, of `nacc` accumulators `acc_stride` TMEM columns apart
// (nacc = 0: this CTA had no K blocks, the result is zero).  `ok` must be
// warp-uniform.  With `stage` (free shared memory, 4 KB per warpgroup), the
// direct path goes through shared memory so that C is written in 16-byte
// pieces of whole rows instead of one 2-byte value per thread and row.
template <bool BF16, int BLOCK_M, int DQ_WG>
__device__ __forceinline__ void tc_epilogue(const GemmArgs &p, uint32_t d_addr, int wg, int dw,
                                            int lane, int r, int n0, int m0, int split, bool ok,
                                            int nacc, uint32_t acc_stride, int *last_flag,
                                            uint8_t *stage = nullptr) {
  constexpr int DQ_THREADS = 128 * DQ_WG;
  const int N = p.N, M = p.M;
  const int n = n0 + r;
  const bool direct = (p.splits == 1);
  if (ok) {
    // warpgroups take alternate 16-column chunks of D
    for (int c0 = wg * 16; c0 < BLOCK_M; c0 += 16 * DQ_WG) {
      if (m0 + c0 >= M) break;  // warp-uniform
      float x16[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) x16[j] = 0.f;
      for (int a = 0; a < nacc; ++a) {
        uint32_t v[16];
        __syncwarp();
        tmem_ld_16(d_addr + a * acc_stride + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) x16[j] = a == 0 ? __uint_as_float(v[j]) : x16[j] + __uint_as_float(v[j]);
      }
      if (direct && stage != nullptr) {
        // [16 rows][128 columns] of 16-bit values; thread r writes column r,
        // then each thread copies two 16-byte pieces of whole rows to C
        uint16_t *T = reinterpret_cast<uint16_t *>(stage + wg * 4096);
#pragma unroll
        for (int j = 0; j < 16; ++j) T[j * 128 + r] = f32_to_16<BF16>(x16[j]);
        named_bar_sync(2 + wg, 128);
#pragma unroll
        for (int q = r; q < 256; q += 128) {
          const int row = q >> 4, col = (q & 15) * 8;
          const int m = m0 + c0 + row;
          if (m < M)
            *reinterpret_cast<uint4 *>(p.C + static_cast<size_t>(m) * N + n0 + col) =
                *reinterpret_cast<const uint4 *>(T + row * 128 + col);
        }
        named_bar_sync(2 + wg, 128);
        continue;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = m0 + c0 + j;
        if (m < M) {
          const float x = x16[j];
          if (direct)
            p.C[static_cast<size_t>(m) * N + n] = f32_to_16<BF16>(x);
          else
            p.ws[(static_cast<size_t>(split) * M + m) * N + n] = x;
        }
      }
    }
  }
  if (direct) return;
  // the barrier orders every epilogue thread's partial writes before one
  // thread's release-acquire arrival on the tile counter (cumulative
  // release); the second barrier passes the acquire on to all of them
  named_bar_sync(1, DQ_THREADS);
  unsigned int *ctr = p.counters + (static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x);
  if (dw == 0 && lane == 0) {
    const unsigned prev = atomic_add_acq_rel_gpu(ctr, 1u);
    *last_flag = (prev == static_cast<unsigned>(p.splits - 1));
  }
  named_bar_sync(1, DQ_THREADS);
  if (!*last_flag) return;
  // fixed split order per element; 8 independent loads in flight
  const size_t split_stride = static_cast<size_t>(M) * N;
  for (int c = wg; c < BLOCK_M; c += DQ_WG) {
    const int m = m0 + c;
    if (m >= M) break;
    const float *src = p.ws + static_cast<size_t>(m) * N + n;
    float acc = 0.f;
    int sp = 0;
    for (; sp + 8 <= p.splits; sp += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + (sp + j) * split_stride);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc += v[j];
    }
    for (; sp < p.splits; ++sp) acc += __ldcg(src + sp * split_stride);
    p.C[static_cast<size_t>(m) * N + n] = f32_to_16<BF16>(acc);
  }
  if (dw == 0 && lane == 0) *ctr = 0u;
}

}  // namespace tmw4

// gemv.cu -- split-K GEMV for small M on the CUDA cores.
//
// Each CTA owns one 64-column strip of the packed weight (one atom column)
// and one K range.  Its eight warps stream whole 2 KB atoms with 128-bit
// non-coherent loads (512 contiguous bytes per warp instruction: coalesced,
// pith.science review, Figure 22), dequantize in registers exactly as the
// dequant-only kernel does, and accumulate in fp32 against activations held
// in shared memory (mixed-precision fp16/bf16 x fp16/bf16 -> fp32 FMAs).  Partials of the eight warps are summed in a fixed order;
// with split-K, partials go to the workspace and the last CTA of a strip to
// arrive sums them in split order, so results do not depend on scheduling.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "dequant.cuh"
#include "kernels.h"
#include "mma_frag.cuh"

namespace tmw4 {

template <bool BF16>
__device__ __forceinline__ uint16_t float_to_16(float x) {
  if constexpr (BF16) {
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&b);
  } else {
    __half h = __float2half_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
  }
}

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

constexpr int GEMV_WARPS = 8;

// acc += w.lo * a.lo + w.hi * a.hi with fp32 accumulation, for packed 16-bit
// pairs w and a.  The mixed-precision FMA multiplies the two 16-bit inputs
// exactly (at most 22 significant bits) and rounds once into fp32, exactly as
// converting both to fp32 and using an fp32 FMA would.
template <bool BF16>
__device__ __forceinline__ float fma_pair(uint32_t w, uint32_t a, float acc) {
  float r;
  if constexpr (BF16) {
    asm("{\n\t.reg .b16 wl, wh, al, ah;\n\t"
        "mov.b32 {wl, wh}, %1;\n\tmov.b32 {al, ah}, %2;\n\t"
        "fma.rn.f32.bf16 %0, wl, al, %3;\n\t"
        "fma.rn.f32.bf16 %0, wh, ah, %0;\n\t}"
        : "=f"(r) : "r"(w), "r"(a), "f"(acc));
  } else {
    asm("{\n\t.reg .f16 wl, wh, al, ah;\n\t"
        "mov.b32 {wl, wh}, %1;\n\tmov.b32 {al, ah}, %2;\n\t"
        "fma.rn.f32.f16 %0, wl, al, %3;\n\t"
        "fma.rn.f32.f16 %0, wh, ah, %0;\n\t}"
        : "=f"(r) : "r"(w), "r"(a), "f"(acc));
  }
  return r;
}

// The end of a GEMV CTA: red[warp][m][64] holds each warp's sums of rows
// m < MT of the CTA's 64-column strip (after a CTA barrier).  They are added
// in warp order; without split-K the result goes to C, with split-K to the
// workspace, and the last CTA of the strip to arrive adds the splits' partials
// in split order (the counter is reset for the next launch).
template <bool BF16, int MT>
__device__ __forceinline__ void gemv_epilogue(const GemmArgs &p, const float *red, int na, int split, int tid) {
  const int M = p.M, N = p.N;
  __shared__ int s_last;
  // thread t handles outputs (m, cl) = divmod(t + 256 i, 64), i = 0..MT/4
  constexpr int PER_THREAD = (MT * 64 + 255) / 256;
  float sum[PER_THREAD];
#pragma unroll
  for (int i = 0; i < PER_THREAD; ++i) {
    const int idx = tid + 256 * i;
    sum[i] = 0.f;
    if (idx < MT * 64) {
      const int m = idx / 64, cl = idx % 64;
#pragma unroll
      for (int w = 0; w < GEMV_WARPS; ++w) sum[i] += red[(w * MT + m) * 64 + cl];
    }
  }
  if (p.splits == 1) {
#pragma unroll
    for (int i = 0; i < PER_THREAD; ++i) {
      const int idx = tid + 256 * i, m = idx / 64, n = na * ATOM_N + idx % 64;
      if (idx < MT * 64 && m < M) p.C[static_cast<size_t>(m) * N + n] = float_to_16<BF16>(sum[i]);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < PER_THREAD; ++i) {
    const int idx = tid + 256 * i, m = idx / 64, n = na * ATOM_N + idx % 64;
    if (idx < MT * 64 && m < M) p.ws[(static_cast<size_t>(split) * M + m) * N + n] = sum[i];
  }
  // the barrier orders the CTA's partial writes before one thread's
  // release-acquire arrival on the strip counter (cumulative release); the
  // second barrier passes the acquire on to the whole CTA
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomic_add_acq_rel_gpu(p.counters + na, 1u);
    s_last = (prev == static_cast<unsigned>(p.splits - 1));
  }
  __syncwarp();   // lane 0 of warp 0 must be out of its branch before the barrier
  __syncthreads();
  if (!s_last) return;
#pragma unroll
  for (int i = 0; i < PER_THREAD; ++i) {
    const int idx = tid + 256 * i, m = idx / 64, n = na * ATOM_N + idx % 64;
    if (idx < MT * 64 && m < M) {
      // fixed split order (this CTA's own partial from registers); eight
      // independent loads in flight
      const float *src = p.ws + static_cast<size_t>(m) * N + n;
      const size_t stride = static_cast<size_t>(M) * N;
      float t = 0.f;
      int s0 = 0;
      for (; s0 + 8 <= p.splits; s0 += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = s0 + j == split ? sum[i] : __ldcg(src + (s0 + j) * stride);
#pragma unroll
        for (int j = 0; j < 8; ++j) t += v[j];
      }
      for (; s0 < p.splits; ++s0) t += s0 == split ? sum[i] : __ldcg(src + s0 * stride);
      p.C[static_cast<size_t>(m) * N + n] = float_to_16<BF16>(t);
    }
  }
  if (tid == 0) p.counters[na] = 0u;
}

template <bool BF16, int MT>
__global__ void __launch_bounds__(256) gemv_kernel(GemmArgs p) {
  extern __shared__ float4 smem_f4[];
  float *red = reinterpret_cast<float *>(smem_f4);          // [GEMV_WARPS][MT][64]
  uint16_t *As = reinterpret_cast<uint16_t *>(red + GEMV_WARPS * MT * 64);  // [MT][ldA]
  const int na = blockIdx.x, split = blockIdx.y;
  const int KB = p.K / ATOM_K;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(KB, kb0 + p.kb_per_split);
  const int ldA = p.kb_per_split * ATOM_K;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int M = p.M, N = p.N;

  float acc[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;

  const int nA = na * ATOM_N + lane, nB = nA + 32;
  const int G_rows = p.K / p.group;
  // register double buffer: the next atom's four 128-bit loads and its raw
  // scale and zero bytes are in flight while the current atom is
  // dequantized; nothing consumes a loaded value before its atom's turn, so
  // no load stalls the warp early
  // sc/zb[h][col]: scale and zero byte of column nA (col 0) / nB (col 1) for
  // the atom's 32-K half h (the same group unless G = 32)
  uint4 cur[4], nxt[4];
  uint16_t sc_c[2][2], sc_n[2][2];
  uint8_t zb_c[2][2], zb_n[2][2];
  const bool has_zeros = p.zeros != nullptr;
  auto fetch = [&](int kb, uint4 (&c)[4], uint16_t (&sc)[2][2], uint8_t (&zb)[2][2]) {
    const uint4 *atom = reinterpret_cast<const uint4 *>(p.qw + atom_offset(kb, na, KB));
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = ldg_stream(atom + lane + 32 * i);
    const int g = (kb * ATOM_K) / p.group;
    sc[0][0] = __ldg(p.scales + scale_index(g, nA, G_rows));
    sc[0][1] = __ldg(p.scales + scale_index(g, nB, G_rows));
    zb[0][0] = has_zeros ? __ldg(p.zeros + zero_byte(g, nA, G_rows)) : static_cast<uint8_t>(0x88u);
    zb[0][1] = has_zeros ? __ldg(p.zeros + zero_byte(g, nB, G_rows)) : static_cast<uint8_t>(0x88u);
    if (p.group == 32) {   // the second 32-K half has a group of its own
      sc[1][0] = __ldg(p.scales + scale_index(g + 1, nA, G_rows));
      sc[1][1] = __ldg(p.scales + scale_index(g + 1, nB, G_rows));
      zb[1][0] = has_zeros ? __ldg(p.zeros + zero_byte(g + 1, nA, G_rows)) : static_cast<uint8_t>(0x88u);
      zb[1][1] = has_zeros ? __ldg(p.zeros + zero_byte(g + 1, nB, G_rows)) : static_cast<uint8_t>(0x88u);
    } else {
      sc[1][0] = sc[0][0];
      sc[1][1] = sc[0][1];
      zb[1][0] = zb[0][0];
      zb[1][1] = zb[0][1];
    }
  };
  const int zsh = (lane & 1) * 4;   // nA and nB = nA + 32 have the same parity
  int kb = kb0 + warp;
  // the packed weights do not depend on earlier kernels in the stream: the
  // first atom's loads go out before waiting for them
  if (kb < kb1) fetch(kb, cur, sc_c, zb_c);
  pdl_wait();
  pdl_launch_dependents();

  // activations of this K range -> shared memory, 16 bytes per copy (rows >= M are zero)
  const int klen = (kb1 - kb0) * ATOM_K;
  for (int idx = tid; idx < MT * (klen / 8); idx += blockDim.x) {
    const int m = idx / (klen / 8), kk = (idx % (klen / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m < M)
      v = *reinterpret_cast<const uint4 *>(p.A + static_cast<size_t>(m) * p.K + kb0 * ATOM_K + kk);
    *reinterpret_cast<uint4 *>(As + m * ldA + kk) = v;
  }
  __syncwarp();   // a CTA barrier counts a warp as arrived once any lane reaches it
  __syncthreads();

  for (; kb < kb1; kb += GEMV_WARPS) {
    const int kbn = kb + GEMV_WARPS;
    if (kbn < kb1) fetch(kbn, nxt, sc_n, zb_n);
    uint32_t s2c[2][2], zmc[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        s2c[h][i] = dup16(sc_c[h][i]);
        zmc[h][i] = zero_magic2<BF16>((static_cast<uint32_t>(zb_c[h][i]) >> zsh) & 0xFu);
      }
#pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
      const int col = ci & 1, h = ci >> 1;
      const uint32_t w[4] = {cur[ci].x, cur[ci].y, cur[ci].z, cur[ci].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t d[4];
        dequant_word<BF16>(w[j], zmc[h][col], s2c[h][col], d);
        const int kloc = (kb - kb0) * ATOM_K + 32 * h + 8 * j;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint4 av = *reinterpret_cast<const uint4 *>(As + m * ldA + kloc);
          float s = acc[m][ci];
          s = fma_pair<BF16>(d[0], av.x, s);
          s = fma_pair<BF16>(d[1], av.y, s);
          s = fma_pair<BF16>(d[2], av.z, s);
          s = fma_pair<BF16>(d[3], av.w, s);
          acc[m][ci] = s;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        sc_c[h][i] = sc_n[h][i];
        zb_c[h][i] = zb_n[h][i];
      }
  }
  // per-warp partials -> shared memory, then a fixed-order sum over warps
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    red[(warp * MT + m) * 64 + lane] = acc[m][0] + acc[m][2];
    red[(warp * MT + m) * 64 + lane + 32] = acc[m][1] + acc[m][3];
  }
  __syncthreads();
  gemv_epilogue<BF16, MT>(p, red, na, split, tid);
}


// ----------------------------------------------------------- 8-bit weights
// The same CTA structure for 8-bit codes (int8 with byte zeros, or FP8 E4M3;
// GemmArgs::fp8): a strip's 64-K atom is half of an 8 KB tile block, lane l
// again owns columns nA = 64 na + l and nB = nA + 32 and loads their 64 K as
// 4 + 4 chunks of 16 consecutive K (512 contiguous bytes per warp
// instruction); each word of 4 codes becomes two pairs w = T(s * v)
// (dequant.cuh) and meets the activations in mixed-precision FMAs.
template <bool BF16, int MT>
__global__ void __launch_bounds__(256) gemv8_kernel(GemmArgs p) {
  extern __shared__ float4 smem_f4[];
  float *red = reinterpret_cast<float *>(smem_f4);          // [GEMV_WARPS][MT][64]
  uint16_t *As = reinterpret_cast<uint16_t *>(red + GEMV_WARPS * MT * 64);  // [MT][ldA]
  const int na = blockIdx.x, split = blockIdx.y;
  const int KB = p.K / ATOM_K;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(KB, kb0 + p.kb_per_split);
  const int ldA = p.kb_per_split * ATOM_K;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int M = p.M;
  const bool fp8 = p.fp8 != 0;

  float acc[MT][2];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = 0.f;

  const int nA = na * ATOM_N + lane, nB = nA + 32;
  const int G_rows = p.K / p.group;
  const bool has_zeros = p.zeros != nullptr;
  // cur/nxt[2 kq + col]: chunk kq (16 K) of column nA (col 0) / nB (col 1);
  // sc/zb[h][col]: scale and zero of the atom's 32-K half h
  uint4 cur[8], nxt[8];
  uint16_t sc_c[2][2], sc_n[2][2];
  uint8_t zb_c[2][2], zb_n[2][2];
  auto zero8 = [&](int g, int n) -> uint8_t {
    return has_zeros ? __ldg(p.zeros + (static_cast<size_t>(n >> 7) * G_rows + g) * TILE_N + (n & 127))
                     : static_cast<uint8_t>(128u);
  };
  auto fetch = [&](int kb, uint4 (&c)[8], uint16_t (&sc)[2][2], uint8_t (&zb)[2][2]) {
    const uint8_t *blk = p.qw + (static_cast<size_t>(na >> 1) * KB + kb) * (2 * BLOCK_BYTES) + (na & 1) * ATOM_N * 16;
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
      const uint4 *row = reinterpret_cast<const uint4 *>(blk + kq * 2048);
      c[2 * kq] = ldg_stream(row + lane);
      c[2 * kq + 1] = ldg_stream(row + lane + 32);
    }
    const int g = (kb * ATOM_K) / p.group;
    sc[0][0] = __ldg(p.scales + scale_index(g, nA, G_rows));
    sc[0][1] = __ldg(p.scales + scale_index(g, nB, G_rows));
    zb[0][0] = zero8(g, nA);
    zb[0][1] = zero8(g, nB);
    if (p.group == 32) {   // the second 32-K half has a group of its own
      sc[1][0] = __ldg(p.scales + scale_index(g + 1, nA, G_rows));
      sc[1][1] = __ldg(p.scales + scale_index(g + 1, nB, G_rows));
      zb[1][0] = zero8(g + 1, nA);
      zb[1][1] = zero8(g + 1, nB);
    } else {
      sc[1][0] = sc[0][0];
      sc[1][1] = sc[0][1];
      zb[1][0] = zb[0][0];
      zb[1][1] = zb[0][1];
    }
  };
  int kb = kb0 + warp;
  if (kb < kb1) fetch(kb, cur, sc_c, zb_c);
  pdl_wait();
  pdl_launch_dependents();

  // activations of this K range -> shared memory, 16 bytes per copy (rows >= M are zero)
  const int klen = (kb1 - kb0) * ATOM_K;
  for (int idx = tid; idx < MT * (klen / 8); idx += blockDim.x) {
    const int m = idx / (klen / 8), kk = (idx % (klen / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m < M)
      v = *reinterpret_cast<const uint4 *>(p.A + static_cast<size_t>(m) * p.K + kb0 * ATOM_K + kk);
    *reinterpret_cast<uint4 *>(As + m * ldA + kk) = v;
  }
  __syncwarp();   // a CTA barrier counts a warp as arrived once any lane reaches it
  __syncthreads();

  for (; kb < kb1; kb += GEMV_WARPS) {
    const int kbn = kb + GEMV_WARPS;
    if (kbn < kb1) fetch(kbn, nxt, sc_n, zb_n);
    uint32_t s2c[2][2], zmc[2][2];
    float sfc[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        s2c[h][i] = dup16(sc_c[h][i]);
        zmc[h][i] = zero_magic2<false>(zb_c[h][i]);
        sfc[h][i] = BF16 ? __uint_as_float(static_cast<uint32_t>(sc_c[h][i]) << 16)
                         : __half2float(__ushort_as_half(sc_c[h][i]));
      }
#pragma unroll
    for (int ci = 0; ci < 8; ++ci) {
      const int kq = ci >> 1, col = ci & 1, h = kq >> 1;
      const uint32_t w[4] = {cur[ci].x, cur[ci].y, cur[ci].z, cur[ci].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t d[2];
        dequant_word8<BF16>(w[j], fp8, zmc[h][col], zb_c[h][col], s2c[h][col], sfc[h][col], d);
        const int kloc = (kb - kb0) * ATOM_K + 16 * kq + 4 * j;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint2 av = *reinterpret_cast<const uint2 *>(As + m * ldA + kloc);
          float s = acc[m][col];
          s = fma_pair<BF16>(d[0], av.x, s);
          s = fma_pair<BF16>(d[1], av.y, s);
          acc[m][col] = s;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        sc_c[h][i] = sc_n[h][i];
        zb_c[h][i] = zb_n[h][i];
      }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    red[(warp * MT + m) * 64 + lane] = acc[m][0];
    red[(warp * MT + m) * 64 + lane + 32] = acc[m][1];
  }
  __syncthreads();
  gemv_epilogue<BF16, MT>(p, red, na, split, tid);
}

// ----------------------------------------------------------- tensor-core mode
// The same CTA structure (one 64-column strip, one K range, eight warps
// taking its 64-K atoms in turn, partials in warp then split order), with the
// multiply-accumulate on the tensor cores: each thread loads exactly its
// mma.sync m16n8k16 A fragments of an atom from global memory (8-byte
// pieces; 2 x 128 contiguous bytes per warp instruction), turns the codes
// into exact (q - z) 16-bit values, multiplies them with the activations (B
// fragments from a 128-byte-swizzled shared copy: conflict-free) and scales
// the atom's fp32 sums by the group scale, C += s * sum_k a_k (q_k - z).
// The CUDA-core kernel above spends one FMA per weight per row; this one
// one MMA per eight weights for up to 8 NT8 rows.
//
// Fragment roles: A = weights (m16 tile mt: strip columns 16 mt + g and
// 16 mt + 8 + g), B = activations (n8 tile j8: rows 8 j8 + g), K order within
// a 64-K atom permuted alike on both sides: thread (g, t) holds K
// [16t, 16t + 16) -- half of one 16-byte chunk of a column.
constexpr int GEMV_MMA_RED_FLOATS = GEMV_WARPS * 16 * 64;   // [warp][16 rows][64 columns]

// Shared memory of the tensor-core mode for `kb_per_split` atoms per split:
// the reduction area, the activations [kb][8 NT8 rows][128 B] (swizzled),
// the strip's scales [groups][64] and zero bytes [groups][32].
__host__ __device__ constexpr size_t gemv_mma_smem(int nt8, int kb_per_split, int group) {
  return sizeof(float) * GEMV_MMA_RED_FLOATS + 1024 + static_cast<size_t>(kb_per_split) * 1024 * nt8 +
         static_cast<size_t>((kb_per_split * ATOM_K) / group + 2) * (128 + 32);
}

__device__ __forceinline__ uint2 ldg_stream_u2(const void *p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

template <bool BF16, int NT8>
__global__ void __launch_bounds__(256, 2) gemv_mma_kernel(GemmArgs p) {
  extern __shared__ float4 smem_f4[];
  float *red = reinterpret_cast<float *>(smem_f4);                        // [warp][16][64]
  uint8_t *act = align_smem_1024(reinterpret_cast<uint8_t *>(red + GEMV_MMA_RED_FLOATS));
  const int na = blockIdx.x, split = blockIdx.y;
  const int KB = p.K / ATOM_K;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(KB, kb0 + p.kb_per_split);
  const int nkb = kb1 - kb0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int M = p.M;
  const int G_rows = p.K / p.group;
  const int g_lo = (kb0 * ATOM_K) / p.group;
  const int ng = ((kb1 * ATOM_K - 1) / p.group) - g_lo + 1;              // groups the range meets
  uint16_t *sc_s = reinterpret_cast<uint16_t *>(act + static_cast<size_t>(nkb) * 1024 * NT8);   // [ng][64]
  uint8_t *zb_s = reinterpret_cast<uint8_t *>(sc_s + ng * 64);                                   // [ng][32]
  const bool has_zeros = p.zeros != nullptr;

  // this thread's A pieces of an atom: column 16 mt + 8 h + g, K [16t, 16t + 16)
  const int piece = (t >> 1) * 1024 + g * 16 + (t & 1) * 8;
  uint2 cur[4][2], nxt[4][2];
  auto fetch = [&](int kb, uint2 (&w)[4][2]) {
    const uint8_t *atom = p.qw + atom_offset(kb, na, KB) + piece;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) w[mt][h] = ldg_stream_u2(atom + (16 * mt + 8 * h) * 16);
  };
  int kb = kb0 + warp;
  // the packed weights do not depend on earlier kernels in the stream: the
  // first atom's loads go out before waiting for them
  if (kb < kb1) fetch(kb, cur);
  pdl_wait();
  pdl_launch_dependents();

  // activations of the K range, rows >= M zero: 16-byte chunk c of row m of
  // atom j at act + j 1024 NT8 + m 128 + ((c ^ (m % 8)) << 4)
  for (int idx = tid; idx < nkb * 8 * NT8 * 8; idx += blockDim.x) {
    const int c = idx & 7, m = (idx >> 3) % (8 * NT8), j = (idx >> 3) / (8 * NT8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m < M) v = *reinterpret_cast<const uint4 *>(p.A + static_cast<size_t>(m) * p.K + (kb0 + j) * ATOM_K + 8 * c);
    *reinterpret_cast<uint4 *>(act + j * 1024 * NT8 + m * 128 + ((c ^ (m & 7)) << 4)) = v;
  }
  // the strip's scales and zero bytes of the groups the range meets
  for (int idx = tid; idx < ng * 64; idx += blockDim.x) {
    const int gi = idx >> 6, cl = idx & 63;
    sc_s[idx] = p.scales[scale_index(g_lo + gi, na * ATOM_N + cl, G_rows)];
    if (has_zeros && (cl & 1) == 0) zb_s[gi * 32 + (cl >> 1)] = p.zeros[zero_byte(g_lo + gi, na * ATOM_N + cl, G_rows)];
  }
  __syncwarp();
  __syncthreads();

  float acc[4][NT8][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][j8][e] = 0.f;
  int brd[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) brd[i] = g * 128 + (((2 * t + (i >> 1)) ^ g) << 4) + ((i & 1) << 3);
  const int zsh = (g & 1) * 4;   // columns 16 mt + 8 h + g have the parity of g

  for (; kb < kb1; kb += GEMV_WARPS) {
    const int kbn = kb + GEMV_WARPS;
    if (kbn < kb1) fetch(kbn, nxt);
    // the atom's group: scales and (MAGIC + z), -(64 + z) per column
    const int gi = (kb * ATOM_K) / p.group - g_lo;
    float sc[4][2];
    uint32_t zm[4][2], z16[4][2];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int cl = 16 * mt + 8 * h + g;
        sc[mt][h] = bits16_to_f32<BF16>(sc_s[gi * 64 + cl]);
        const uint32_t z = has_zeros ? (static_cast<uint32_t>(zb_s[gi * 32 + (cl >> 1)]) >> zsh) & 0xFu : 8u;
        zm[mt][h] = z * 0x00010001u + Magic<BF16>::pair;
        z16[mt][h] = z * 0x00100010u + 0xD400D400u;
      }
    float accg[4][NT8][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
        for (int e = 0; e < 4; ++e) accg[mt][j8][e] = 0.f;
    const uint8_t *ast = act + (kb - kb0) * 1024 * NT8;
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
      uint2 bf[NT8][2];
#pragma unroll
      for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
        for (int j = 0; j < 2; ++j) bf[j8][j] = *reinterpret_cast<const uint2 *>(ast + j8 * 1024 + brd[2 * wi + j]);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t lo[4], hi[4];
        codes_minus_zero<BF16>(wi == 0 ? cur[mt][0].x : cur[mt][0].y, zm[mt][0], z16[mt][0], lo);
        codes_minus_zero<BF16>(wi == 0 ? cur[mt][1].x : cur[mt][1].y, zm[mt][1], z16[mt][1], hi);
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int j8 = 0; j8 < NT8; ++j8)
            mma_16816<BF16>(accg[mt][j8], lo[2 * j], hi[2 * j], lo[2 * j + 1], hi[2 * j + 1], bf[j8][j].x,
                            bf[j8][j].y);
      }
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int j8 = 0; j8 < NT8; ++j8) {
        ffma2(acc[mt][j8][0], acc[mt][j8][1], sc[mt][0], sc[mt][0], accg[mt][j8][0], accg[mt][j8][1]);
        ffma2(acc[mt][j8][2], acc[mt][j8][3], sc[mt][1], sc[mt][1], accg[mt][j8][2], accg[mt][j8][3]);
      }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) cur[mt][h] = nxt[mt][h];
  }
  // per-warp sums -> red[warp][m][64]: element e of (mt, j8) is row
  // m = 8 j8 + 2t + e % 2, strip column 16 mt + 8 (e / 2) + g
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int j8 = 0; j8 < NT8; ++j8)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        red[(warp * 8 * NT8 + 8 * j8 + 2 * t + (e & 1)) * 64 + 16 * mt + 8 * (e >> 1) + g] = acc[mt][j8][e];
  __syncthreads();
  gemv_epilogue<BF16, 8 * NT8>(p, red, na, split, tid);
}

size_t gemv_smem_bytes(int rows_tmpl, int kb_per_split) {
  return sizeof(float) * static_cast<size_t>(GEMV_WARPS) * rows_tmpl * 64 +
         sizeof(uint16_t) * static_cast<size_t>(rows_tmpl) * kb_per_split * ATOM_K;
}

template <bool BF16, int MT>
static cudaError_t launch_gemv_t(const GemmArgs &a, cudaStream_t st) {
  const size_t smem = gemv_smem_bytes(MT, a.kb_per_split);   // at most 200 KB (checked by the caller)
  cudaError_t e = smem_optin<gemv_kernel<BF16, MT>>(200 * 1024);
  if (e != cudaSuccess) return e;
  dim3 grid(a.N / ATOM_N, a.splits);
  return launch_kernel(gemv_kernel<BF16, MT>, grid, dim3(256), smem, st, a.pdl != 0, a);
}

size_t gemv_mma_smem_bytes(int nt8, int kb_per_split, int group) { return gemv_mma_smem(nt8, kb_per_split, group); }

template <bool BF16, int NT8>
static cudaError_t launch_gemv_mma_t(const GemmArgs &a, cudaStream_t st) {
  const size_t smem = gemv_mma_smem(NT8, a.kb_per_split, a.group);   // at most 200 KB (checked by the caller)
  cudaError_t e = smem_optin<gemv_mma_kernel<BF16, NT8>>(200 * 1024);
  if (e != cudaSuccess) return e;
  dim3 grid(a.N / ATOM_N, a.splits);
  return launch_kernel(gemv_mma_kernel<BF16, NT8>, grid, dim3(256), smem, st, a.pdl != 0, a);
}

template <bool BF16, int MT>
static cudaError_t launch_gemv8_t(const GemmArgs &a, cudaStream_t st) {
  const size_t smem = gemv_smem_bytes(MT, a.kb_per_split);   // at most 200 KB (checked by the caller)
  cudaError_t e = smem_optin<gemv8_kernel<BF16, MT>>(200 * 1024);
  if (e != cudaSuccess) return e;
  dim3 grid(a.N / ATOM_N, a.splits);
  return launch_kernel(gemv8_kernel<BF16, MT>, grid, dim3(256), smem, st, a.pdl != 0, a);
}

cudaError_t launch_gemv(const GemmArgs &a, bool bf16, int rows_tmpl, bool mma, cudaStream_t st) {
  if (a.wbits == 8) {
    switch (rows_tmpl) {
      case 1: return bf16 ? launch_gemv8_t<true, 1>(a, st) : launch_gemv8_t<false, 1>(a, st);
      case 2: return bf16 ? launch_gemv8_t<true, 2>(a, st) : launch_gemv8_t<false, 2>(a, st);
      case 4: return bf16 ? launch_gemv8_t<true, 4>(a, st) : launch_gemv8_t<false, 4>(a, st);
      case 8: return bf16 ? launch_gemv8_t<true, 8>(a, st) : launch_gemv8_t<false, 8>(a, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (mma) {
    switch (rows_tmpl) {
      case 8: return bf16 ? launch_gemv_mma_t<true, 1>(a, st) : launch_gemv_mma_t<false, 1>(a, st);
      case 16: return bf16 ? launch_gemv_mma_t<true, 2>(a, st) : launch_gemv_mma_t<false, 2>(a, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (rows_tmpl) {
    case 1: return bf16 ? launch_gemv_t<true, 1>(a, st) : launch_gemv_t<false, 1>(a, st);
    case 2: return bf16 ? launch_gemv_t<true, 2>(a, st) : launch_gemv_t<false, 2>(a, st);
    case 4: return bf16 ? launch_gemv_t<true, 4>(a, st) : launch_gemv_t<false, 4>(a, st);
    case 8: return bf16 ? launch_gemv_t<true, 8>(a, st) : launch_gemv_t<false, 8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tmw4

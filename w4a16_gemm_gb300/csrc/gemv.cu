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
  uint4 cur[4], nxt[4];
  uint16_t sc_c[2], sc_n[2];
  uint8_t zb_c[2], zb_n[2];
  const bool has_zeros = p.zeros != nullptr;
  auto fetch = [&](int kb, uint4 (&c)[4], uint16_t (&sc)[2], uint8_t (&zb)[2]) {
    const uint4 *atom = reinterpret_cast<const uint4 *>(p.qw + atom_offset(kb, na, KB));
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = ldg_stream(atom + lane + 32 * i);
    const int g = (kb * ATOM_K) / p.group;
    sc[0] = __ldg(p.scales + scale_index(g, nA, G_rows));
    sc[1] = __ldg(p.scales + scale_index(g, nB, G_rows));
    zb[0] = has_zeros ? __ldg(p.zeros + zero_byte(g, nA, G_rows)) : static_cast<uint8_t>(0x88u);
    zb[1] = has_zeros ? __ldg(p.zeros + zero_byte(g, nB, G_rows)) : static_cast<uint8_t>(0x88u);
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
    uint32_t s2c[2], zmc[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      s2c[i] = dup16(sc_c[i]);
      zmc[i] = zero_magic2<BF16>((static_cast<uint32_t>(zb_c[i]) >> zsh) & 0xFu);
    }
#pragma unroll
    for (int ci = 0; ci < 4; ++ci) {
      const int col = ci & 1, h = ci >> 1;
      const uint32_t w[4] = {cur[ci].x, cur[ci].y, cur[ci].z, cur[ci].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t d[4];
        dequant_word<BF16>(w[j], zmc[col], s2c[col], d);
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
    for (int i = 0; i < 2; ++i) {
      sc_c[i] = sc_n[i];
      zb_c[i] = zb_n[i];
    }
  }
  // per-warp partials -> shared memory, then a fixed-order sum over warps
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    red[(warp * MT + m) * 64 + lane] = acc[m][0] + acc[m][2];
    red[(warp * MT + m) * 64 + lane + 32] = acc[m][1] + acc[m][3];
  }
  __syncthreads();
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

cudaError_t launch_gemv(const GemmArgs &a, bool bf16, int rows_tmpl, cudaStream_t st) {
  switch (rows_tmpl) {
    case 1: return bf16 ? launch_gemv_t<true, 1>(a, st) : launch_gemv_t<false, 1>(a, st);
    case 2: return bf16 ? launch_gemv_t<true, 2>(a, st) : launch_gemv_t<false, 2>(a, st);
    case 4: return bf16 ? launch_gemv_t<true, 4>(a, st) : launch_gemv_t<false, 4>(a, st);
    case 8: return bf16 ? launch_gemv_t<true, 8>(a, st) : launch_gemv_t<false, 8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tmw4

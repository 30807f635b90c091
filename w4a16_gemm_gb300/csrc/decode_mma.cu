// decode_mma.cu -- split-K streaming kernel for small row counts (M <= 32)
// whose multiply-accumulate runs on the tensor cores with register operands.
//
// At decode sizes the GEMM is bound by HBM, and with the dequantization
// spread over many threads the SM's instruction issue is the next limit:
// every instruction spent per packed 32-bit word (eight weights) lowers the
// bandwidth a full GPU can sustain.  This kernel therefore keeps the
// per-word work minimal:
//   * each thread streams its own 8-byte slices of the packed blocks with
//     64-bit non-coherent loads (a warp instruction covers two whole
//     128-byte lines), DM_DEPTH 64-K blocks ahead, straight into registers;
//   * codes become (q - z) exactly in 16-bit floats (exponent-magic OR,
//     then one exact subtract; TurboMind paper, pith.science review,
//     Figure 6: integer-to-float conversion before the scaling);
//   * the registers feed mma.sync m16n8k16 directly as its A operand (16
//     weight columns x 16 K), the activations are the B operand (8 rows per
//     n8 tile), and the fp32 accumulator of one quantization group is scaled
//     once per group: C += s * sum_k a_k (q_k - z).  With s applied in fp32
//     the only roundings are those of the fp32 sums and the final one to the
//     16-bit output.
// The K order inside each MMA is a permutation of the actual K order that
// both operands share: thread (g, t) of the fragment layout holds, for
// every column it owns, the 16 consecutive K values [16t, 16t + 16) of a
// 64-K block -- exactly half of one 16-byte chunk of the packed layout (a
// chunk is 32 consecutive K of one column) -- and the activations are read
// with the same mapping.  No shuffle is needed on either side.
//
// CTA: 4 warps, one 128-column tile of the packed weight, one K range
// (split-K over grid.y).  Warp w owns columns 32w + 8j + g (j = 0..3; two
// m16 tiles: rows g / g+8 of tile 0 are columns g / g+8, of tile 1 columns
// g+16 / g+24).  Activations of the CTA's K range are staged once in shared
// memory (rows M..8*NT8-1 zero).  With split-K, fp32 partials go to the
// workspace and the last CTA of a tile to arrive adds them in split order,
// so results do not depend on scheduling.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tmw4_device.cuh"

namespace tmw4 {

namespace {

constexpr int DM_THREADS = 128;
constexpr int DM_DEPTH = 8;      // ring slots per warp: up to DM_DEPTH - 1 blocks in flight
constexpr int DM_SLOT = 1024;    // one warp's share of a 64-K block: 32 columns x 32 bytes
constexpr int DM_META = 80;      // a group's scales (64 B) and zeros (16 B) for one warp

// 16-byte asynchronous copy global -> shared (cached in L2 only).  The
// copies of one thread are committed in groups and waited for with
// cp.async.wait_group; the data is visible to the copying thread after the
// wait, and to the rest of its warp after a following __syncwarp.
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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

// Shared memory of a CTA:
//   weight ring   [warp][DM_DEPTH][c 0..3][lane][8 B]: slot r of warp w holds
//                 the warp's 1 KB of one 64-K block, the 8 bytes each lane
//                 consumes at [c][lane] (filled by 16-byte copies that span
//                 two neighbouring lanes);
//   group data    [warp][DM_DEPTH][80 B]: scales of the warp's 32 columns
//                 (64 B) and their zero nibbles (16 B), in the slot of the
//                 block that starts the group;
//   activations   one 16-byte A-fragment quad per (m16 tile, 16-K step,
//                 lane): {a[g][K..K+1], a[g+8][K..K+1], a[g][K+2..K+3],
//                 a[g+8][K+2..K+3]} with K = 16t + 4i inside 64-K block kb
//                 (i = step within the block), in lane order, so a warp's
//                 128-bit read is 512 contiguous bytes.
constexpr int DM_RING_BYTES = 4 * DM_DEPTH * (DM_SLOT + DM_META);

size_t decode_mma_smem_bytes(int nt16, int kb_per_split) {
  return DM_RING_BYTES + static_cast<size_t>(nt16) * kb_per_split * 4 * 32 * 16;
}

// NT16: m16 tiles of activation rows (M <= 16 * NT16).  GS: 64-K blocks per
// quantization group (1 for G = 64, 2 for G = 128); kb_per_split is a
// multiple of GS, so every split starts on a group boundary.
//
// Fragment roles (mma.sync m16n8k16, row.col): A = activations (16 rows x 16
// K), B = dequantized weights (16 K x 8 columns), D = C^T tile in fp32.
// Thread (g, t) = (lane / 4, lane % 4) holds B column g: for K step i of a
// 64-K block, b0 = pair (16t + 4i, +1) and b1 = pair (16t + 4i + 2, +3) of
// that column -- the pairs 2(i%2) and 2(i%2)+1 of word i/2 of its 8-byte
// slice -- and the A quad above, so both operands see the same K order.
template <bool BF16, int NT16, int GS>
__global__ void __launch_bounds__(DM_THREADS) decode_mma_kernel(GemmArgs p) {
  extern __shared__ uint4 dm_smem[];
  constexpr int D = DM_DEPTH;
  static_assert(D % GS == 0, "group starts must fall on fixed ring slots");
  const int nt = blockIdx.x, split = blockIdx.y;
  const int KB = p.K / 64;
  const int kb0 = split * p.kb_per_split;
  const int nsteps = min(KB, kb0 + p.kb_per_split) - kb0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G_rows = p.K / p.group;
  const int KS = 4 * p.kb_per_split;          // 16-K steps of a full split
  const bool has_zeros = p.zeros != nullptr;

  uint8_t *smem = reinterpret_cast<uint8_t *>(dm_smem);
  const uint32_t ring = smem_u32(smem) + warp * D * DM_SLOT;                       // slot r: + r * DM_SLOT
  const uint32_t meta = smem_u32(smem) + 4 * D * DM_SLOT + warp * D * DM_META;     // slot r: + r * DM_META
  const uint8_t *meta_p = smem + 4 * D * DM_SLOT + warp * D * DM_META;
  uint4 *act = reinterpret_cast<uint4 *>(smem + DM_RING_BYTES);

  // copies of block s (relative to kb0): lane (g, h, e) = (L/4, (L/2)%2, L%2)
  // copies the 16-byte chunk half h of column 32w + 8c + g for c = 2e, 2e+1
  // into [c][lanes 4g + 2h, +1] of the slot
  const int h_cp = (lane >> 1) & 1, e_cp = lane & 1;
  const uint8_t *wsrc = p.qw + (static_cast<size_t>(nt) * KB + kb0) * BLOCK_BYTES + (warp >> 1) * ATOM_BYTES +
                        h_cp * 1024 + ((warp & 1) * 32 + 16 * e_cp + g) * 16;
  const uint32_t wdst = ring + (2 * e_cp) * 256 + 32 * g + 16 * h_cp;
  // group u of the split: lanes 0-3 copy the warp's 64 bytes of scales
  // (columns 32w + 8q .. +8, q = lane), lane 4 its 16 zero bytes
  const uint8_t *msrc =
      lane < 4 ? reinterpret_cast<const uint8_t *>(p.scales + (static_cast<size_t>(nt) * G_rows + kb0 / GS) * TILE_N +
                                                   32 * warp + 8 * lane)
               : (lane == 4 && has_zeros
                      ? p.zeros + (static_cast<size_t>(nt) * G_rows + kb0 / GS) * (TILE_N / 2) + 16 * warp
                      : nullptr);
  const size_t mstride = lane < 4 ? TILE_N * 2 : TILE_N / 2;    // bytes per group
  const uint32_t mdst = meta + (lane < 4 ? 16 * lane : 64);

  auto issue = [&](int s) {
    if (s < nsteps) {
      const int r = s % D;
      const uint8_t *src = wsrc + static_cast<size_t>(s) * BLOCK_BYTES;
      cp_async16(wdst + r * DM_SLOT, src);
      cp_async16(wdst + r * DM_SLOT + 256, src + 128);
      if (s % GS == 0 && msrc != nullptr) cp_async16(mdst + r * DM_META, msrc + (s / GS) * mstride);
    }
    cp_async_commit();   // one group per block, empty past the end
  };

  // the packed weights do not depend on earlier kernels in the stream: the
  // first blocks are requested before waiting for them
#pragma unroll
  for (int s = 0; s < D - 1; ++s) issue(s);
  pdl_wait();
  pdl_launch_dependents();

  // activations of this K range -> interleaved A quads (rows >= M are zero).
  // Lane (g, t) of warp w fills, for every half block hb (32 K) with
  // hb % 4 == w, the quads of 16-K steps 2hb and 2hb + 1 of its own fragment
  // position: one 16-byte load per row covers both.
#pragma unroll
  for (int mt = 0; mt < NT16; ++mt) {
    const int m0 = 16 * mt + g, m1 = m0 + 8;
    const uint16_t *r0 = p.A + static_cast<size_t>(m0) * p.K + kb0 * 64 + 16 * t;
    const uint16_t *r1 = p.A + static_cast<size_t>(m1) * p.K + kb0 * 64 + 16 * t;
    const bool has0 = m0 < p.M, has1 = m1 < p.M;
    for (int hb = warp; hb < 2 * nsteps; hb += 4) {
      // 16-K steps 2hb and 2hb + 1 of this lane start at K = 64 (hb / 2) + 16t + 8 (hb % 2) and 4 later
      const int koff = (hb >> 1) * 64 + (hb & 1) * 8;
      uint4 u = make_uint4(0u, 0u, 0u, 0u), v = make_uint4(0u, 0u, 0u, 0u);
      if (has0) u = *reinterpret_cast<const uint4 *>(r0 + koff);
      if (has1) v = *reinterpret_cast<const uint4 *>(r1 + koff);
      uint4 *dst = act + (mt * KS + 2 * hb) * 32 + lane;
      dst[0] = make_uint4(u.x, v.x, u.y, v.y);
      dst[32] = make_uint4(u.z, v.z, u.w, v.w);
    }
  }
  __syncthreads();

  float acc[NT16][4][4];
  float accg[NT16][4][4];
#pragma unroll
  for (int mt = 0; mt < NT16; ++mt)
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][c][e] = 0.f;

  uint32_t zm[4], z16[4];   // per column of the current group: (MAGIC + z), -(64 + z) (fp16)
  float sc_lo[4], sc_hi[4]; // per column pair of the current group: the scales
  const int zsh = (g >> 1) * 8 + (g & 1) * 4;
  const uint2 *wread = reinterpret_cast<const uint2 *>(smem + warp * D * DM_SLOT) + lane;   // + r*128 + c*32
  const uint4 *aq = act + lane;               // A quad of 16-K step ks: aq[ks * 32]

#pragma unroll 1
  for (int s0 = 0; s0 < nsteps; s0 += D) {
#pragma unroll
    for (int r = 0; r < D; ++r) {
      const int s = s0 + r;
      if (s >= nsteps) break;
      // block s has landed (at most D - 2 younger groups pending) and every
      // lane is past its reads of the slot refilled next (block s - 1)
      cp_async_wait<D - 2>();
      __syncwarp();
      issue(s + D - 1);
      uint2 w[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) w[c] = wread[r * (DM_SLOT / 8) + c * 32];
      if (r % GS == 0) {
        // group start: its scales and zero points
        const uint8_t *m = meta_p + r * DM_META;
        const uint4 zw = has_zeros ? *reinterpret_cast<const uint4 *>(m + 64) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t sp2 = *reinterpret_cast<const uint32_t *>(m + 16 * c + 4 * t);
          sc_lo[c] = bits16_to_f32<BF16>(sp2 & 0xFFFFu);
          sc_hi[c] = bits16_to_f32<BF16>(sp2 >> 16);
          const uint32_t zwc = c == 0 ? zw.x : c == 1 ? zw.y : c == 2 ? zw.z : zw.w;
          const uint32_t z = has_zeros ? (zwc >> zsh) & 0xFu : 8u;
          zm[c] = z * 0x00010001u + Magic<BF16>::pair;
          z16[c] = z * 0x00100010u + 0xD400D400u;   // fp16 -(64 + z) in both halves
        }
#pragma unroll
        for (int mt = 0; mt < NT16; ++mt)
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) accg[mt][c][e] = 0.f;
      }
#pragma unroll
      for (int wi = 0; wi < 2; ++wi) {
        uint32_t bq[4][4];
#pragma unroll
        for (int c = 0; c < 4; ++c) codes_minus_zero<BF16>(wi == 0 ? w[c].x : w[c].y, zm[c], z16[c], bq[c]);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int mt = 0; mt < NT16; ++mt) {
            const uint4 a = aq[(mt * KS + 4 * s + 2 * wi + j) * 32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
              mma_16816<BF16>(accg[mt][c], a.x, a.y, a.z, a.w, bq[c][2 * j], bq[c][2 * j + 1]);
          }
        }
      }
      if (r % GS == GS - 1) {
        // end of a group: C += s * sum over the group
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int mt = 0; mt < NT16; ++mt) {
            ffma2(acc[mt][c][0], acc[mt][c][1], sc_lo[c], sc_hi[c], accg[mt][c][0], accg[mt][c][1]);
            ffma2(acc[mt][c][2], acc[mt][c][3], sc_lo[c], sc_hi[c], accg[mt][c][2], accg[mt][c][3]);
          }
      }
    }
  }
  cp_async_wait<0>();

  // accumulator element e of (mt, c): row m = 16 mt + g + 8 (e >> 1),
  // column n = 128 nt + 32 w + 8 c + 2t + (e & 1); elements e and e + 1 are
  // two adjacent columns of one row
  const int M = p.M, N = p.N;
  const int nbase = nt * TILE_N + 32 * warp + 2 * t;
  if (p.splits == 1) {
#pragma unroll
    for (int mt = 0; mt < NT16; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int m = 16 * mt + g + 8 * h;
          const int n = nbase + 8 * c;
          if (m < M)
            *reinterpret_cast<uint32_t *>(p.C + static_cast<size_t>(m) * N + n) =
                static_cast<uint32_t>(f32_to_bits16<BF16>(acc[mt][c][2 * h])) |
                (static_cast<uint32_t>(f32_to_bits16<BF16>(acc[mt][c][2 * h + 1])) << 16);
        }
    return;
  }
#pragma unroll
  for (int mt = 0; mt < NT16; ++mt)
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int m = 16 * mt + g + 8 * h;
        const int n = nbase + 8 * c;
        if (m < M)
          *reinterpret_cast<float2 *>(p.ws + (static_cast<size_t>(split) * M + m) * N + n) =
              make_float2(acc[mt][c][2 * h], acc[mt][c][2 * h + 1]);
      }
  // the barrier orders the CTA's partial writes before one thread's
  // release-acquire arrival on the tile counter (cumulative release); the
  // second barrier passes the acquire on to the whole CTA
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomic_add_acq_rel_gpu(p.counters + nt, 1u);
    s_last = (prev == static_cast<unsigned>(p.splits - 1));
  }
  __syncwarp();
  __syncthreads();
  if (!s_last) return;
  const size_t stride = static_cast<size_t>(M) * N;
#pragma unroll
  for (int mt = 0; mt < NT16; ++mt)
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int m = 16 * mt + g + 8 * h;
        const int n = nbase + 8 * c;
        if (m < M) {
          // fixed split order; this CTA's own partial from registers
          const float2 *src = reinterpret_cast<const float2 *>(p.ws + static_cast<size_t>(m) * N + n);
          const float2 mine = make_float2(acc[mt][c][2 * h], acc[mt][c][2 * h + 1]);
          float2 sum = make_float2(0.f, 0.f);
          int q0 = 0;
          for (; q0 + 8 <= p.splits; q0 += 8) {
            float2 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = q0 + q == split ? mine : __ldcg(src + (q0 + q) * stride / 2);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              sum.x += v[q].x;
              sum.y += v[q].y;
            }
          }
          for (; q0 < p.splits; ++q0) {
            const float2 v = q0 == split ? mine : __ldcg(src + q0 * stride / 2);
            sum.x += v.x;
            sum.y += v.y;
          }
          *reinterpret_cast<uint32_t *>(p.C + static_cast<size_t>(m) * N + n) =
              static_cast<uint32_t>(f32_to_bits16<BF16>(sum.x)) |
              (static_cast<uint32_t>(f32_to_bits16<BF16>(sum.y)) << 16);
        }
      }
  if (threadIdx.x == 0) p.counters[nt] = 0u;
}

template <bool BF16, int NT16, int GS>
static cudaError_t launch_dm_t(const GemmArgs &a, cudaStream_t st) {
  auto kern = decode_mma_kernel<BF16, NT16, GS>;
  cudaError_t e = smem_optin<decode_mma_kernel<BF16, NT16, GS>>(static_cast<int>(kDecodeMmaMaxSmem));
  if (e != cudaSuccess) return e;
  const size_t smem = decode_mma_smem_bytes(NT16, a.kb_per_split);
  dim3 grid(a.N / TILE_N, a.splits);
  return launch_kernel(kern, grid, dim3(DM_THREADS), smem, st, a.pdl != 0, a);
}

template <bool BF16, int NT16>
static cudaError_t launch_dm_g(const GemmArgs &a, cudaStream_t st) {
  return a.group == 64 ? launch_dm_t<BF16, NT16, 1>(a, st) : launch_dm_t<BF16, NT16, 2>(a, st);
}

int decode_mma_nt16(int M) { return M <= 16 ? 1 : M <= 32 ? 2 : 0; }

cudaError_t launch_decode_mma(const GemmArgs &a, bool bf16, cudaStream_t st) {
  switch (decode_mma_nt16(a.M)) {
    case 1: return bf16 ? launch_dm_g<true, 1>(a, st) : launch_dm_g<false, 1>(a, st);
    case 2: return bf16 ? launch_dm_g<true, 2>(a, st) : launch_dm_g<false, 2>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tmw4

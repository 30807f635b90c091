// attn_decode.cu -- decode attention (one query token per sequence) over a
// low-bit KV cache: the attention pipeline of the TurboMind paper
// (pith.science review, Figure 4: the low-bit cache is loaded, converted to
// 16-bit values by integer-to-float conversion and scaling, and multiplied
// in Q K^T and P V on tensor cores; Figure 10: the cache is consumed in
// 64-token tiles whose loads overlap the two products).
//
//   K[t, d] = T(ks[t] * (kq[t, d] - kz[t])),  V likewise   (per token, KV head)
//   O[hq]   = softmax_t(sm_scale * Q[hq] . K[t]) V,  t < len,  h = hq / GQ
//
// Blackwell form:
//   - A persistent grid takes units (sequence b, KV head h, chunk c of up to
//     chunk_tiles 64-token tiles) from a ticket counter, one at a time, over
//     a per-sequence prefix of unit counts that every CTA scans into shared
//     memory.  One producer lane streams each tile's K and V rows with TMA
//     tensor copies (128-byte swizzle for 8-bit rows, 64-byte for 4-bit rows,
//     so the transposing reads below hit distinct banks), the tile's scales
//     and zeros with bulk copies and, for a unit's first tile, the group's
//     queries, into a ring whose stages also carry the unit's description.
//   - Four consumer warps take 16 tokens of each tile.  S^T = Q K^T runs on
//     mma.sync m16n8k16 with the query heads as the 16 rows (GQ <= 16) and
//     exact (q - z) keys as the B operand; the head dimension is summed in a
//     permuted order (any order gives the same sum) chosen so that each
//     thread's B fragments come from contiguous bytes of one key row.  The
//     per-token key scale multiplies the fp32 scores, which feed an online
//     softmax (exp2, running max and sum per head); P' = P * (value scale),
//     rounded to 16 bits, is the A operand of O += P' (q - z), whose B
//     fragments pair two tokens of one value column: the byte permute that
//     builds them is the "transpose V" step of Figure 4, done in registers.
//   - At a unit's end the four warps merge through shared memory; a unit
//     that covers its whole sequence writes O, otherwise it leaves (m, l, O)
//     in a workspace slot and the last chunk to arrive (one acq_rel atomic)
//     merges the chunks in order.  Every wait is bounded (the consumer warps'
//     own barrier is an mbarrier for that reason).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "mma_frag.cuh"
#include "ptx.cuh"

namespace tmw4 {
namespace {

constexpr int AD_D = 128;     // head dimension
constexpr int AD_TT = 64;     // tokens per tile (one ring stage)
constexpr int AD_CW = 4;      // consumer warps; warp w takes tokens 16w..16w+15 of a tile
constexpr int AD_THREADS = 32 * (AD_CW + 1);
constexpr int AD_CSTRIDE = AD_D + 4;   // floats per row of the merge area
// CTAs per SM the register allocation targets with at most 8 query heads per
// KV head (a build option: -DTMW4_AD_MINB=n)
#ifndef TMW4_AD_MINB
#define TMW4_AD_MINB 2
#endif
constexpr int AD_SLOT = AD_D + 4;      // floats per workspace slot: O[128], m, l, pad (16-byte rows)

template <int BITS>
struct AdGeom {
  static constexpr int ROW = AD_D * BITS / 8;                  // bytes per cached token row
  static constexpr int KV = AD_TT * ROW;                       // one K (or V) tile
  static constexpr int PRM = AD_TT * 2 * 2 + AD_TT * 2;        // ks, vs (16-bit), kz, vz (bytes)
  static constexpr int TX = 2 * KV + PRM;                      // bytes landing per stage
  static constexpr int META = 2 * KV + 512 - 128;              // 8 ints: the stage's unit and tile
  static constexpr int QOFF = 2 * KV + 512;                    // a unit's queries (first tile only)
  static constexpr int QMAX = 16 * AD_D * 2;                   // at most 16 query heads
  static constexpr int STAGE = ((QOFF + QMAX + 1023) / 1024) * 1024;
  static constexpr int NS = BITS == 8 ? 3 : 5;                 // ring stages
  static constexpr int RING = NS * STAGE;
};

// What a ring stage holds (written by the producer before it arms the
// stage's barrier, read by the consumers after it completes).
struct AdMeta {
  int b, h, c, tt;     // sequence, KV head, chunk, tile within the chunk
  int ntile, nch;      // tiles of this unit (0: empty sequence), chunks of the sequence
  int len, end;        // sequence length; end = 1: no more units
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&r);
  } else {
    const __half2 r = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&r);
  }
}

// Cached codes become exact (q - z) values in 16 bits; the per-token scales
// are applied to fp32 quantities instead: to the scores (S = s_t * sum_d
// Q_d (q - z)) and to the probabilities that multiply the values
// (P'_t = P_t * s_t, rounded once to 16 bits for the MMA).  With P = 1 (a
// single token) the output is RNE(s * (q - z)) exactly, as in the
// definition; otherwise it differs from dequantizing first only by rounding
// (it skips the rounding of each s * (q - z) to 16 bits).
//   fp16 codes: the byte under the exponent magic 0x6400 is 1024 + q
//   exactly; minus (1024 + z) is exact.  bf16 8-bit codes: 2^23 + q in fp32,
//   minus 2^23 + z, converted exactly (|q - z| <= 255 fits 8 bits).  4-bit
//   codes: codes_minus_zero.
constexpr uint32_t kMagic16 = 0x64646464u;

__device__ __forceinline__ uint32_t sub_f16x2(uint32_t x, uint32_t zm) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(zm));
  return r;
}

// fp32 value of byte e of w, exactly: 2^23 + byte
__device__ __forceinline__ float byte_f32(uint32_t w, int e) {
  return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | e));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One key word (four codes of one token): (q - z) pairs (e0, e1), (e2, e3).
template <bool BF16>
__device__ __forceinline__ void k8_diff(uint32_t w, uint32_t zm, float zf, uint32_t &p01, uint32_t &p23) {
  if constexpr (BF16) {
    (void)zm;
    p01 = pack2<true>(byte_f32(w, 0) - zf, byte_f32(w, 1) - zf);
    p23 = pack2<true>(byte_f32(w, 2) - zf, byte_f32(w, 3) - zf);
  } else {
    (void)zf;
    p01 = sub_f16x2(__byte_perm(w, kMagic16, 0x4140), zm);
    p23 = sub_f16x2(__byte_perm(w, kMagic16, 0x4342), zm);
  }
}

// Two value words of tokens a and b (same four columns): p[e] = (column e
// of a, column e of b) as (q - z), each with its own token's zero.
template <bool BF16>
__device__ __forceinline__ void v8_diff(uint32_t a, uint32_t b, uint32_t zm, float za, float zb,
                                        uint32_t (&p)[4]) {
  if constexpr (BF16) {
    (void)zm;
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = pack2<true>(byte_f32(a, e) - za, byte_f32(b, e) - zb);
  } else {
    (void)za;
    (void)zb;
    const uint32_t t01 = __byte_perm(a, b, 0x5140);   // a.b0, b.b0, a.b1, b.b1
    const uint32_t t23 = __byte_perm(a, b, 0x7362);   // a.b2, b.b2, a.b3, b.b3
    p[0] = sub_f16x2(__byte_perm(t01, kMagic16, 0x4140), zm);
    p[1] = sub_f16x2(__byte_perm(t01, kMagic16, 0x4342), zm);
    p[2] = sub_f16x2(__byte_perm(t23, kMagic16, 0x4140), zm);
    p[3] = sub_f16x2(__byte_perm(t23, kMagic16, 0x4342), zm);
  }
}

// mma_16816 when rows 8..15 of A are zero (at most 8 query heads): those
// rows' accumulators are neither read nor kept, so they take no registers.
template <bool BF16>
__device__ __forceinline__ void mma_16816_lo(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  float x2, x3;
  if constexpr (BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %5}, {%7, %8}, {%9, %10, %11, %11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(x2), "=f"(x3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(b0), "r"(b1), "f"(d[0]), "f"(d[1]), "f"(0.f));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %5}, {%7, %8}, {%9, %10, %11, %11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(x2), "=f"(x3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(b0), "r"(b1), "f"(d[0]), "f"(d[1]), "f"(0.f));
  }
  (void)x2;
  (void)x3;
}

template <bool BF16, bool HI>
__device__ __forceinline__ void mma_q(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                      uint32_t b0, uint32_t b1) {
  if constexpr (HI) {
    mma_16816<BF16>(d, a0, a1, a2, a3, b0, b1);
  } else {
    (void)a1;
    (void)a3;
    mma_16816_lo<BF16>(d, a0, a2, b0, b1);
  }
}

// -(64 + za), -(64 + zb) as an fp16 pair (4-bit codes, fp16 only): exact.
__device__ __forceinline__ uint32_t z16_pair(uint32_t za, uint32_t zb) {
  const __half2 h = __floats2half2_rn(-(64.f + static_cast<float>(za)), -(64.f + static_cast<float>(zb)));
  return *reinterpret_cast<const uint32_t *>(&h);
}

// (magic + za, magic + zb) as a 16-bit pair: exact integers in either type.
template <bool BF16, int BITS>
__device__ __forceinline__ uint32_t zero_pair(uint32_t za, uint32_t zb) {
  if constexpr (BF16 && BITS == 4) {
    return (0x4300u + za) | ((0x4300u + zb) << 16);   // 128 + z, z <= 15: mantissa bits
  } else {
    return (0x6400u + za) | ((0x6400u + zb) << 16);   // 1024 + z, z <= 255
  }
}

template <bool BF16, int BITS, bool HI>
__global__ void __launch_bounds__(AD_THREADS, HI ? 1 : TMW4_AD_MINB)
    attn_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const AttnArgs p) {
  using Gm = AdGeom<BITS>;
  constexpr int NS = Gm::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *ring = align_smem_1024(smem_raw);
  const int GQ = p.Hq / p.Hkv;
  float *cO = reinterpret_cast<float *>(ring + Gm::RING);               // [CW][GQ][CSTRIDE]
  float *cM = cO + AD_CW * GQ * AD_CSTRIDE;                             // [CW][GQ]
  float *cL = cM + AD_CW * GQ;                                          // [CW][GQ]
  uint64_t *full = reinterpret_cast<uint64_t *>(cL + AD_CW * GQ + 2);   // 536 GQ + 2 floats in: 8-byte aligned
  uint64_t *empty = full + NS;
  uint64_t *cbar = empty + NS;                                          // the consumer warps' barrier
  volatile int *flags = reinterpret_cast<volatile int *>(cbar + 1);     // abort, last arriver
  int *wsum = const_cast<int *>(flags) + 2;                             // [AD_CW + 1] warp totals
  int *pref = wsum + AD_CW + 2;                                         // [B + 1] first unit of each sequence
  int *slen = pref + p.B + 1;                                           // [B] clamped lengths

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < NS) {
    mbar_init(full + threadIdx.x, 1);
    mbar_init(empty + threadIdx.x, AD_CW);
  }
  if (threadIdx.x == 0) {
    mbar_init(cbar, AD_CW);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  // the lengths, queries, cache and work tickets may come from the previous kernel
  pdl_wait();
  volatile int *abort_flag = flags;
  const int ctok = p.chunk_tiles * AD_TT;
  unsigned int *ticket = p.counters + static_cast<size_t>(p.B) * p.Hkv;   // next unit; then CTAs finished

  // Units in sequence-major order (sequence b, then chunk, then KV head):
  // sequence b's first unit pref[b], by a block-wide scan of its unit
  // count Hkv * chunks(b) (a sequence of length 0 keeps one chunk, which
  // writes its zero output).
  {
    const int per = (p.B + AD_THREADS - 1) / AD_THREADS;
    const int b0 = min(p.B, static_cast<int>(threadIdx.x) * per), b1 = min(p.B, b0 + per);
    auto units_of = [&](int len) { return p.Hkv * (len == 0 ? 1 : (len + ctok - 1) / ctok); };
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      int len = __ldg(p.lens + b);
      len = len < 0 ? 0 : (len > p.L_max ? p.L_max : len);
      slen[b] = len;
      sum += units_of(len);
    }
    int x = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += wsum[w];
    int run = base + x - sum;
    for (int b = b0; b < b1; ++b) {
      pref[b] = run;
      run += units_of(slen[b]);
    }
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w = 0; w <= AD_CW; ++w) tot += wsum[w];
      pref[p.B] = tot;
    }
    __syncthreads();
  }

  if (warp == AD_CW) {
    // ------------------------------------------------------------ producer
    // Units are handed out by a ticket counter, so that every CTA takes the
    // next unit as soon as it has issued its last one.
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      const int total = pref[p.B];
      int i = 0;
      bool ok = true;
      unsigned int next = atomicAdd(ticket, 1u);
      auto stage_free = [&](int idx) {
        return idx < NS || mbar_wait_idle(empty + idx % NS, ((idx / NS) & 1) ^ 1u, p.limit_ns, abort_flag, p.err,
                                          SITE_PRODUCER_EMPTY, idx, 256);
      };
      while (ok) {
        if (next >= static_cast<unsigned>(total)) break;
        const int u = static_cast<int>(next);
        // the sequence of unit u: the last b with pref[b] <= u
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (pref[mid] <= u) lo = mid; else hi = mid - 1;
        }
        const int cb = lo, len_b = slen[cb];
        const int nch_b = len_b == 0 ? 1 : (len_b + ctok - 1) / ctok;
        const int r = u - pref[cb];
        const int c = r / p.Hkv, h = r % p.Hkv;
        const int t0 = c * ctok;
        const int ntile = len_b == 0 ? 0 : min(p.chunk_tiles, (len_b - t0 + AD_TT - 1) / AD_TT);
        const long long row = (static_cast<long long>(cb) * p.Hkv + h) * p.L_max + t0;
        for (int tt = 0; tt < max(ntile, 1); ++tt, ++i) {
          if (!stage_free(i)) {
            ok = false;
            break;
          }
          const int s = i % NS;
          uint8_t *st = ring + s * Gm::STAGE;
          AdMeta *m = reinterpret_cast<AdMeta *>(st + Gm::META);
          m->b = cb; m->h = h; m->c = c; m->tt = tt;
          m->ntile = ntile; m->nch = nch_b; m->len = len_b; m->end = 0;
          if (ntile == 0) {
            mbar_arrive(full + s);   // no data: the consumers write the zero output
            continue;
          }
          const long long rr = row + static_cast<long long>(tt) * AD_TT;
          const int qbytes = tt == 0 ? GQ * AD_D * 2 : 0;
          mbar_arrive_expect_tx(full + s, Gm::TX + qbytes);
          tma_load_2d(st, &kmap, 0, static_cast<int32_t>(rr), full + s);
          tma_load_2d(st + Gm::KV, &vmap, 0, static_cast<int32_t>(rr), full + s);
          tma_bulk_g2s(st + 2 * Gm::KV, p.k_scale + rr, AD_TT * 2, full + s);
          tma_bulk_g2s(st + 2 * Gm::KV + AD_TT * 2, p.v_scale + rr, AD_TT * 2, full + s);
          tma_bulk_g2s(st + 2 * Gm::KV + AD_TT * 4, p.k_zero + rr, AD_TT, full + s);
          tma_bulk_g2s(st + 2 * Gm::KV + AD_TT * 5, p.v_zero + rr, AD_TT, full + s);
          if (qbytes)
            tma_bulk_g2s(st + Gm::QOFF, p.q + (static_cast<size_t>(cb) * p.Hq + static_cast<size_t>(h) * GQ) * AD_D,
                         qbytes, full + s);
        }
        // the next ticket once this unit is issued (not earlier: a CTA that
        // held a second ticket while others had none would run two units)
        next = atomicAdd(ticket, 1u);
      }
      // the end marker
      if (ok && stage_free(i)) {
        const int s = i % NS;
        reinterpret_cast<AdMeta *>(ring + s * Gm::STAGE + Gm::META)->end = 1;
        mbar_arrive(full + s);
        ++i;
      }
      // every copy issued must land before the CTA exits
      for (int j = max(0, i - NS); j < i; ++j)
        mbar_wait_bounded(full + j % NS, (j / NS) & 1, p.limit_ns, nullptr, p.err, SITE_DRAIN_TMA, j);
    }
  } else {
  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int ctid = threadIdx.x;   // 0..127
  const float NEG_INF = -__int_as_float(0x7F800000);
  uint32_t cphase = 0;
  // barrier of the four consumer warps (an mbarrier, so that its wait is
  // bounded like every other)
  auto cbar_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(cbar);
    const bool okb = mbar_wait_all_idle(cbar, cphase, p.limit_ns, abort_flag, p.err, SITE_DQ_AEMPTY, 0, 64);
    cphase ^= 1u;
    return okb;
  };
  uint32_t qa[8][2], qb[8][2];
  float m_run[2], l_run[2];
  float o[16][4];
  for (int i = 0;; ++i) {
    const int s = i % NS;
    if (!mbar_wait_all_idle(full + s, (i / NS) & 1, p.limit_ns, abort_flag, p.err, SITE_DQ_FULL, i, 128)) break;
    const uint8_t *st = ring + s * Gm::STAGE;
    const AdMeta x = *reinterpret_cast<const AdMeta *>(st + Gm::META);
    if (x.end) break;
    const long long bh = static_cast<long long>(x.b) * p.Hkv + x.h;
    const size_t orow0 = (static_cast<size_t>(x.b) * p.Hq + static_cast<size_t>(x.h) * GQ);
    if (x.ntile == 0) {
      // empty sequence: zero output
      for (int e = ctid; e < GQ * AD_D; e += 32 * AD_CW) p.o[orow0 * AD_D + e] = 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
      continue;
    }
    if (x.tt == 0) {
      // a new unit: Q fragments from the stage (thread t's head-dimension
      // range is [32t, 32t + 32); the order inside it matches the B
      // fragments built from the key rows below), fresh softmax state
      const uint16_t *sq = reinterpret_cast<const uint16_t *>(st + Gm::QOFF);
      uint32_t h0[16], h1[16];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int head = g + 8 * r;
        uint32_t *hv = r == 0 ? h0 : h1;
        if ((r == 0 || HI) && head < GQ) {
          const uint4 *src = reinterpret_cast<const uint4 *>(sq + head * AD_D + 32 * t);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = src[k];
            hv[4 * k] = v.x; hv[4 * k + 1] = v.y; hv[4 * k + 2] = v.z; hv[4 * k + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) hv[k] = 0;
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if constexpr (BITS == 8) {
          // step k: elements 4k, 4k+1 | 4k+2, 4k+3
          qa[k][0] = h0[2 * k]; qa[k][1] = h0[2 * k + 1];
          qb[k][0] = h1[2 * k]; qb[k][1] = h1[2 * k + 1];
        } else {
          // step 2m + r: elements (8m + 2r, 8m + 2r + 4) | (8m + 2r + 1, 8m + 2r + 5)
          const int m = k >> 1, r = k & 1;
          const uint32_t lo0 = h0[4 * m + r], hi0 = h0[4 * m + 2 + r];
          const uint32_t lo1 = h1[4 * m + r], hi1 = h1[4 * m + 2 + r];
          qa[k][0] = __byte_perm(lo0, hi0, 0x5410); qa[k][1] = __byte_perm(lo0, hi0, 0x7632);
          qb[k][0] = __byte_perm(lo1, hi1, 0x5410); qb[k][1] = __byte_perm(lo1, hi1, 0x7632);
        }
      }
      m_run[0] = m_run[1] = NEG_INF;
      l_run[0] = l_run[1] = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
    }
    {
      const uint8_t *sK = st, *sV = st + Gm::KV;
      const uint16_t *sks = reinterpret_cast<const uint16_t *>(st + 2 * Gm::KV);
      const uint16_t *svs = sks + AD_TT;
      const uint8_t *skz = st + 2 * Gm::KV + AD_TT * 4;
      const uint8_t *svz = skz + AD_TT;
      const int tb = 16 * warp;
      const int tok0 = x.c * ctok + x.tt * AD_TT + tb;   // sequence position of this warp's first token

      // every token of this warp's slice is inside the sequence (all but
      // the last tile of a unit): no masking
      const bool full = tok0 + 16 <= x.len;

      // ---- S^T = Q K^T over this warp's 16 tokens (two n8 tiles), on exact
      // (q - z); B-fragment column g of n-tile j is token tb + 8j + g
      float sc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[j][e] = 0.f;
      {
        uint32_t kw[2][8];
        uint32_t kzm[2], kz16[2];
        float kzf[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int r = tb + 8 * j + g;
          const uint32_t z = skz[r];
          kzm[j] = zero_pair<BF16, BITS>(z, z);
          kz16[j] = (BITS == 4 && !BF16) ? z16_pair(z, z) : 0u;
          kzf[j] = __uint_as_float(0x4B000000u | z);
          if constexpr (BITS == 8) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint4 v = *reinterpret_cast<const uint4 *>(sK + r * 128 + (((2 * t + c) ^ (r & 7)) << 4));
              kw[j][4 * c] = v.x; kw[j][4 * c + 1] = v.y; kw[j][4 * c + 2] = v.z; kw[j][4 * c + 3] = v.w;
            }
          } else {
            const uint4 v = *reinterpret_cast<const uint4 *>(sK + r * 64 + ((t ^ ((r >> 1) & 3)) << 4));
            kw[j][0] = v.x; kw[j][1] = v.y; kw[j][2] = v.z; kw[j][3] = v.w;
          }
        }
        if constexpr (BITS == 8) {
#pragma unroll
          for (int s8 = 0; s8 < 8; ++s8)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              uint32_t b0, b1;
              k8_diff<BF16>(kw[j][s8], kzm[j], kzf[j], b0, b1);
              mma_q<BF16, HI>(sc[j], qa[s8][0], qb[s8][0], qa[s8][1], qb[s8][1], b0, b1);
            }
        } else {
          // word m: pairs (8m, 8m+4), (8m+1, 8m+5) feed step 2m; (8m+2, 8m+6),
          // (8m+3, 8m+7) step 2m + 1
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              uint32_t pr[4];
              codes_minus_zero<BF16>(kw[j][m], kzm[j], kz16[j], pr);
              mma_q<BF16, HI>(sc[j], qa[2 * m][0], qb[2 * m][0], qa[2 * m][1], qb[2 * m][1], pr[0], pr[1]);
              mma_q<BF16, HI>(sc[j], qa[2 * m + 1][0], qb[2 * m + 1][0], qa[2 * m + 1][1], qb[2 * m + 1][1], pr[2],
                              pr[3]);
            }
        }
      }

      // ---- scale, mask, online softmax.  Score column e of n-tile j is token
      // tb + 8j + 2t + (e & 1): its key and value scales are read as pairs.
      constexpr int NR = HI ? 2 : 1;   // rows g (and g + 8 with more than 8 heads)
      float kcs[2][2], vsc[2][2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t kp = *reinterpret_cast<const uint32_t *>(sks + tb + 8 * j + 2 * t);
        const uint32_t vp = *reinterpret_cast<const uint32_t *>(svs + tb + 8 * j + 2 * t);
        kcs[j][0] = bits16_to_f32<BF16>(kp & 0xFFFFu) * p.sm_scale_log2;
        kcs[j][1] = bits16_to_f32<BF16>(kp >> 16) * p.sm_scale_log2;
        vsc[j][0] = bits16_to_f32<BF16>(vp & 0xFFFFu);
        vsc[j][1] = bits16_to_f32<BF16>(vp >> 16);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2 * NR; ++e) sc[j][e] *= kcs[j][e & 1];
      if (!full) {
        // a token past the length: score -inf and value scale 0, so that
        // whatever the (unwritten) cache holds there contributes exactly 0
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool valid = tok0 + 8 * j + 2 * t + e < x.len;
            if (!valid) {
              sc[j][e] = NEG_INF;
              if (HI) sc[j][e + 2] = NEG_INF;
              vsc[j][e] = 0.f;
            }
          }
      }
      float pmax[2] = {NEG_INF, NEG_INF};
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2 * NR; ++e) pmax[e >> 1] = fmaxf(pmax[e >> 1], sc[j][e]);
      float corr[2] = {1.f, 1.f}, muse[2] = {0.f, 0.f};
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        pmax[r] = fmaxf(pmax[r], __shfl_xor_sync(0xFFFFFFFFu, pmax[r], 1));
        pmax[r] = fmaxf(pmax[r], __shfl_xor_sync(0xFFFFFFFFu, pmax[r], 2));
        const float mnew = fmaxf(m_run[r], pmax[r]);
        muse[r] = mnew == NEG_INF ? 0.f : mnew;
        corr[r] = ex2(m_run[r] - muse[r]);
        m_run[r] = mnew;
      }
      float psum[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2 * NR; ++e) {
          sc[j][e] = ex2(sc[j][e] - muse[e >> 1]);
          psum[e >> 1] += sc[j][e];
        }
#pragma unroll
      for (int r = 0; r < NR; ++r) l_run[r] = l_run[r] * corr[r] + psum[r];
      if (__any_sync(0xFFFFFFFFu, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
        for (int jn = 0; jn < 16; ++jn) {
          o[jn][0] *= corr[0]; o[jn][1] *= corr[0];
          if constexpr (HI) {
            o[jn][2] *= corr[1]; o[jn][3] *= corr[1];
          }
        }
      }
      // A fragments of P V: P'_t = P_t * s_t (value scale)
      const uint32_t pa0 = pack2<BF16>(sc[0][0] * vsc[0][0], sc[0][1] * vsc[0][1]);
      const uint32_t pa2 = pack2<BF16>(sc[1][0] * vsc[1][0], sc[1][1] * vsc[1][1]);
      const uint32_t pa1 = HI ? pack2<BF16>(sc[0][2] * vsc[0][0], sc[0][3] * vsc[0][1]) : 0u;
      const uint32_t pa3 = HI ? pack2<BF16>(sc[1][2] * vsc[1][0], sc[1][3] * vsc[1][1]) : 0u;

      // ---- O += P' (q - z): B fragments pair tokens (2t, 2t+1) and
      // (2t+8, 2t+9) of value column d = 16 g + jn
      {
        uint32_t vzm[2], vz16[2];
        float vzf[4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t zz = *reinterpret_cast<const uint16_t *>(svz + tb + 8 * h2 + 2 * t);
          const uint32_t za = zz & 0xFFu, zb = zz >> 8;
          vzm[h2] = zero_pair<BF16, BITS>(za, zb);
          vz16[h2] = (BITS == 4 && !BF16) ? z16_pair(za, zb) : 0u;
          vzf[2 * h2] = __uint_as_float(0x4B000000u | za);
          vzf[2 * h2 + 1] = __uint_as_float(0x4B000000u | zb);
        }
        if constexpr (BITS == 8) {
          uint4 vr[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = tb + 2 * t + (q & 1) + 8 * (q >> 1);
            vr[q] = *reinterpret_cast<const uint4 *>(sV + r * 128 + ((g ^ (r & 7)) << 4));
          }
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            uint32_t b0[4], b1[4];
            v8_diff<BF16>((&vr[0].x)[wi], (&vr[1].x)[wi], vzm[0], vzf[0], vzf[1], b0);
            v8_diff<BF16>((&vr[2].x)[wi], (&vr[3].x)[wi], vzm[1], vzf[2], vzf[3], b1);
#pragma unroll
            for (int e = 0; e < 4; ++e) mma_q<BF16, HI>(o[4 * wi + e], pa0, pa1, pa2, pa3, b0[e], b1[e]);
          }
        } else {
          uint2 vr[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = tb + 2 * t + (q & 1) + 8 * (q >> 1);
            vr[q] = *reinterpret_cast<const uint2 *>(sV + r * 64 + ((((g >> 1) ^ ((r >> 1) & 3)) << 4) | ((g & 1) << 3)));
          }
#pragma unroll
          for (int wi = 0; wi < 2; ++wi) {
            // halves from the two tokens: (a.b0, a.b1 | b.b0, b.b1) holds
            // columns 0..3 of both, (a.b2, a.b3 | b.b2, b.b3) columns 4..7
#pragma unroll
            for (int which = 0; which < 2; ++which) {
              const uint32_t sel = which ? 0x7632 : 0x5410;
              uint32_t b0[4], b1[4];
              codes_minus_zero<BF16>(__byte_perm((&vr[0].x)[wi], (&vr[1].x)[wi], sel), vzm[0], vz16[0], b0);
              codes_minus_zero<BF16>(__byte_perm((&vr[2].x)[wi], (&vr[3].x)[wi], sel), vzm[1], vz16[1], b1);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                mma_q<BF16, HI>(o[8 * wi + 4 * which + e], pa0, pa1, pa2, pa3, b0[e], b1[e]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
    if (x.tt != x.ntile - 1) continue;

    // ---- the unit's last tile: merge the four warps
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xFFFFFFFFu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xFFFFFFFFu, l_run[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int head = g + 8 * r;
      if ((r == 0 || HI) && head < GQ) {
        float *row = cO + (warp * GQ + head) * AD_CSTRIDE;
        // fragment order: column n of n-tile jn is value column 16 n + jn
#pragma unroll
        for (int jn = 0; jn < 16; ++jn)
          *reinterpret_cast<float2 *>(row + jn * 8 + 2 * t) = make_float2(o[jn][2 * r], o[jn][2 * r + 1]);
        if (t == 0) {
          cM[warp * GQ + head] = m_run[r];
          cL[warp * GQ + head] = l_run[r];
        }
      }
    }
    if (!cbar_sync()) break;
    const int d = ctid;                              // this thread's value column
    const int fo = (d & 15) * 8 + (d >> 4);          // its place in fragment order
    const bool whole = x.nch == 1;
    float *wsO = p.ws + (static_cast<size_t>(bh) * p.n_chunks_max + x.c) * GQ * AD_SLOT;
    for (int head = 0; head < GQ; ++head) {
      float mx = NEG_INF;
#pragma unroll
      for (int w = 0; w < AD_CW; ++w) mx = fmaxf(mx, cM[w * GQ + head]);
      float acc = 0.f, l = 0.f;
#pragma unroll
      for (int w = 0; w < AD_CW; ++w) {
        const float f = ex2(cM[w * GQ + head] - mx);
        acc += f * cO[(w * GQ + head) * AD_CSTRIDE + fo];
        l += f * cL[w * GQ + head];
      }
      if (whole) {
        reinterpret_cast<uint16_t *>(p.o)[(orow0 + head) * AD_D + d] = f32_to_bits16<BF16>(acc / l);
      } else {
        float *slot = wsO + head * AD_SLOT;
        slot[d] = acc;
        if (d == 0) {
          slot[AD_D] = mx;
          slot[AD_D + 1] = l;
        }
      }
    }
    if (!whole) {
      // publish, count; the last chunk of (b, h) to arrive merges in order
      __threadfence();
      if (!cbar_sync()) break;
      if (ctid == 0) {
        const unsigned old = atomic_add_acq_rel_gpu(p.counters + bh, 1u);
        const bool last = old == static_cast<unsigned>(x.nch - 1);
        if (last) p.counters[bh] = 0;   // self-resetting for the next launch
        flags[1] = last ? 1 : 0;
      }
      if (!cbar_sync()) break;
      if (flags[1]) {
        // warp w merges heads w, w + 4, ...: lane l owns value columns
        // 4l..4l+3; the chunks are read with 16-byte loads, eight in flight
        const float *base = p.ws + static_cast<size_t>(bh) * p.n_chunks_max * GQ * AD_SLOT;
        for (int head = warp; head < GQ; head += AD_CW) {
          float mx = NEG_INF;
#pragma unroll 8
          for (int c = 0; c < x.nch; ++c) mx = fmaxf(mx, __ldcg(base + (c * GQ + head) * AD_SLOT + AD_D));
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          float l = 0.f;
#pragma unroll 8
          for (int c = 0; c < x.nch; ++c) {
            const float *slot = base + (c * GQ + head) * AD_SLOT;
            const float f = ex2(__ldcg(slot + AD_D) - mx);
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(slot) + lane);
            acc.x += f * v.x;
            acc.y += f * v.y;
            acc.z += f * v.z;
            acc.w += f * v.w;
            l += f * __ldcg(slot + AD_D + 1);
          }
          const uint32_t lo = pack2<BF16>(acc.x / l, acc.y / l), hi = pack2<BF16>(acc.z / l, acc.w / l);
          *reinterpret_cast<uint2 *>(p.o + (orow0 + head) * AD_D + 4 * lane) = make_uint2(lo, hi);
        }
      }
    }
    // the merge area and the arrival flag are rewritten by the next unit
    if (!cbar_sync()) break;
  }
  }
  // the last CTA to finish resets the work tickets for the next launch (every
  // producer has taken its last ticket before its CTA gets here)
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned done = atomic_add_acq_rel_gpu(ticket + 1, 1u);
    if (done == gridDim.x - 1) {
      ticket[0] = 0;
      ticket[1] = 0;
    }
  }
}

}  // namespace

size_t attn_decode_smem_bytes(int bits, int gq, int B) {
  const int ring = bits == 8 ? AdGeom<8>::RING : AdGeom<4>::RING;
  const size_t merge = sizeof(float) * (static_cast<size_t>(AD_CW) * gq * AD_CSTRIDE + 2 * AD_CW * gq + 2);
  const int ns = bits == 8 ? AdGeom<8>::NS : AdGeom<4>::NS;
  // barriers, flags, warp totals, unit prefix and lengths
  return 1024 + ring + merge + 16 * ns + 16 + sizeof(int) * (AD_CW + 2 + 2 * static_cast<size_t>(B) + 1);
}

template <bool BF16, int BITS, bool HI>
static cudaError_t launch_ad_t(const CUtensorMap &km, const CUtensorMap &vm, const AttnArgs &a, int grid,
                               cudaStream_t st) {
  auto kern = attn_decode_kernel<BF16, BITS, HI>;
  const size_t smem = attn_decode_smem_bytes(BITS, a.Hq / a.Hkv, a.B);
  cudaError_t e = smem_optin<attn_decode_kernel<BF16, BITS, HI>>(
      static_cast<int>(attn_decode_smem_bytes(BITS, 16, kAttnMaxBatch)));
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(grid), dim3(AD_THREADS), smem, st, a.pdl != 0, km, vm, a);
}

template <bool BF16, int BITS, bool HI>
static int ad_occ_t(int gq, int batch) {
  int n = 0;
  if (smem_optin<attn_decode_kernel<BF16, BITS, HI>>(
          static_cast<int>(attn_decode_smem_bytes(BITS, 16, kAttnMaxBatch))) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_kernel<BF16, BITS, HI>, AD_THREADS,
                                                    attn_decode_smem_bytes(BITS, gq, batch)) != cudaSuccess)
    return 0;
  return n;
}

int attn_decode_ctas_per_sm(bool bf16, int bits, int gq, int batch) {
  const bool hi = gq > 8;
#define AD_OCC(B, W, H) \
  if (bf16 == B && bits == W && hi == H) return ad_occ_t<B, W, H>(gq, batch);
  AD_OCC(false, 8, false) AD_OCC(false, 8, true) AD_OCC(false, 4, false) AD_OCC(false, 4, true)
  AD_OCC(true, 8, false) AD_OCC(true, 8, true) AD_OCC(true, 4, false) AD_OCC(true, 4, true)
#undef AD_OCC
  return 0;
}

cudaError_t launch_attn_decode(const CUtensorMap &kmap, const CUtensorMap &vmap, const AttnArgs &a, bool bf16,
                               int bits, int grid, cudaStream_t st) {
  const bool hi = a.Hq / a.Hkv > 8;
#define AD_LAUNCH(B, W, H) \
  if (bf16 == B && bits == W && hi == H) return launch_ad_t<B, W, H>(kmap, vmap, a, grid, st);
  AD_LAUNCH(false, 8, false) AD_LAUNCH(false, 8, true) AD_LAUNCH(false, 4, false) AD_LAUNCH(false, 4, true)
  AD_LAUNCH(true, 8, false) AD_LAUNCH(true, 8, true) AD_LAUNCH(true, 4, false) AD_LAUNCH(true, 4, true)
#undef AD_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace tmw4

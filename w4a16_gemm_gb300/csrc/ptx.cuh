// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarrier, TMA (bulk and
// tensor), tcgen05 (TMEM alloc/ld/st, MMA, commit, fences), and the bounded
// wait used by every kernel of this library.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "tmw4_device.cuh"

namespace tmw4 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or the hint (ns) runs out, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// `base` (dynamic shared memory) advanced to the next multiple of 1024 bytes
// of the shared window.  Pointer arithmetic on the shared array (not a round
// trip through an integer) lets the compiler keep accesses through the
// result as shared-memory instructions instead of generic ones.
__device__ __forceinline__ uint8_t *align_smem_1024(uint8_t *base) {
  return base + ((1024u - (smem_u32(base) & 1023u)) & 1023u);
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Gives up
// after `limit_ns` (or as soon as *abort becomes non-zero), records
// TM_DEVERR_TIMEOUT in the device error word and returns false.  No wait in
// this library is unbounded.  The first wait to give up on the device also
// records where: err_word[1] = 1, [2] = site, [3] = linear block index,
// [4] = thread index, [5] = the waiter's stage/step index, [6] = parity.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns, volatile int *abort,
                                                  unsigned int *err_word, unsigned site = 0,
                                                  unsigned step = 0,
                                                  unsigned long long *spin = nullptr) {
#ifdef TMW4_TRACE
  // debug builds: spin[0] += calls, spin[1] += polls of the barrier
  if (spin != nullptr) atomicAdd(spin, 1ull);
#else
  (void)spin;
#endif
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#ifdef TMW4_TRACE
    if (spin != nullptr) atomicAdd(spin + 1, 1ull);
#endif
    if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
    {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        if (abort != nullptr) *abort = 1;
        if (err_word != nullptr) {
          atomicOr(err_word, TM_DEVERR_TIMEOUT);
          if (atomicCAS(err_word + 1, 0u, 1u) == 0u) {
            err_word[2] = site;
            err_word[3] = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
            err_word[4] = threadIdx.x;
            err_word[5] = step;
            err_word[6] = parity;
          }
        }
        return false;
      }
    }
  }
}

// Bounded wait that backs off with __nanosleep between polls (32 ns,
// doubling up to max_sleep_ns), so that a waiting warp takes no issue slots
// from the warps it shares a scheduler with.  For a producer whose ring is
// full, or a consumer whose data is late; the other arguments and the
// result are those of mbar_wait_bounded.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                                  volatile int *abort, unsigned int *err_word, unsigned site,
                                                  unsigned step, unsigned max_sleep_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  unsigned ns = 32;
  while (true) {
    __nanosleep(ns);
    ns = ns * 2 < max_sleep_ns ? ns * 2 : max_sleep_ns;
    if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      if (abort != nullptr) *abort = 1;
      if (err_word != nullptr) {
        atomicOr(err_word, TM_DEVERR_TIMEOUT);
        if (atomicCAS(err_word + 1, 0u, 1u) == 0u) {
          err_word[2] = site;
          err_word[3] = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
          err_word[4] = threadIdx.x;
          err_word[5] = step;
          err_word[6] = parity;
        }
      }
      return false;
    }
  }
}

// Waits of a thread (or warp) with nothing else to do meanwhile: a TMA
// producer whose ring is full, or a consumer whose data has not landed.
// With TMW4_WAIT_BACKOFF (the default) they back off with __nanosleep
// (mbar_wait_backoff); built with -DTMW4_WAIT_BACKOFF=0 they poll with
// try_wait like mbar_wait_bounded.  A polling waiter issues an instruction
// every few tens of cycles, taken from the warps that share its scheduler.
#ifndef TMW4_WAIT_BACKOFF
#define TMW4_WAIT_BACKOFF 1
#endif
__device__ __forceinline__ bool mbar_wait_idle(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                               volatile int *abort, unsigned int *err_word, unsigned site,
                                               unsigned step, unsigned max_sleep_ns = 256) {
#if TMW4_WAIT_BACKOFF
  return mbar_wait_backoff(bar, parity, limit_ns, abort, err_word, site, step, max_sleep_ns);
#else
  (void)max_sleep_ns;
  return mbar_wait_bounded(bar, parity, limit_ns, abort, err_word, site, step);
#endif
}

// Warp-wide form (all 32 lanes call it; the result is warp-uniform): one
// poll and one vote when the phase is already complete, else every lane
// that saw it incomplete waits as mbar_wait_idle does.
__device__ __forceinline__ bool mbar_wait_all_idle(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                                   volatile int *abort, unsigned int *err_word, unsigned site,
                                                   unsigned step, unsigned max_sleep_ns = 128) {
  bool ok = mbar_try_wait(bar, parity);
  if (__all_sync(0xFFFFFFFFu, ok)) return true;
  if (!ok) ok = mbar_wait_idle(bar, parity, limit_ns, abort, err_word, site, step, max_sleep_ns);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Warp-wide bounded wait: lane 0 waits (sleeping in hardware), the warp
// agrees on the outcome, then every lane takes its own acquire with one
// non-blocking test of the (now completed) phase.  Must be called by all 32
// lanes.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                               volatile int *abort, unsigned int *err_word,
                                               unsigned site, unsigned step,
                                               unsigned long long *spin = nullptr) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  if (lane == 0) ok = mbar_wait_bounded(bar, parity, limit_ns, abort, err_word, site, step, spin);
  ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  if (ok) (void)mbar_try_wait(bar, parity);
  return ok;
}

// Warp-wide bounded wait in which every lane polls the barrier itself: one
// poll and one vote when the phase is already complete (the common case in
// a pipeline that runs ahead), the bounded loop otherwise.  The result is
// warp-uniform.
__device__ __forceinline__ bool mbar_wait_all(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int *abort, unsigned int *err_word,
                                              unsigned site, unsigned step,
                                              unsigned long long *spin = nullptr) {
  const bool done = mbar_try_wait(bar, parity);
  if (__all_sync(0xFFFFFFFFu, done)) return true;
  const bool ok = done || mbar_wait_bounded(bar, parity, limit_ns, abort, err_word, site, step, spin);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Device-scope atomic add with acquire-release semantics; returns the old value.
__device__ __forceinline__ unsigned atomic_add_acq_rel_gpu(unsigned *addr, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

// ldmatrix .x4: four 8x8 matrices of 16-bit elements from shared memory;
// lane 8m + r gives the address of row r of matrix m (16 bytes, 16-byte
// aligned), and thread (g, t) receives in d[m] the elements (2t, 2t + 1) of
// row g of matrix m.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&d)[4], uint32_t smem_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
               : "r"(smem_addr));
}

// --------------------------------------------------------- thread-block cluster
// Rank of this CTA in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Cluster-wide barrier of all threads of all CTAs of the cluster (release /
// acquire at cluster scope).  Every thread of every CTA must reach it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of `smem_addr` (a shared::cta address) in the
// CTA of the cluster with rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
// Store to the shared memory of a CTA of the cluster (a shared::cluster
// address from mapa_shared).
__device__ __forceinline__ void st_shared_cluster_f32(uint32_t cluster_addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                             uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst_smem, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst_smem, const CUtensorMap *map, int32_t x,
                                            int32_t y, int32_t z, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch (griddepcontrol, sm_90 and later).  A kernel
// launched with programmatic stream serialization may start while the
// previous kernel in the stream is still running.  pdl_wait() blocks the
// calling thread until every kernel this launch depends on has completed and
// its memory writes are visible; it returns at once for a plain launch.
// pdl_launch_dependents() lets the next such launch in the stream start
// early (the next kernel still waits for this one before reading its output).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------- tcgen05
// TMEM addresses: bits [31:16] lane, bits [15:0] column (32-bit cells).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` once all tcgen05 async operations issued so far by this
// thread have completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Four MMAs over one 64-K block: A columns a_tmem + 0/8/16/24 (16 K each),
// B descriptors b_desc + 0/2/4/6 (32 bytes further along K each, in 16-byte
// units of the descriptor's start address).  `first` clears D on the first
// MMA instead of accumulating.
__device__ __forceinline__ void tc_mma_ts_kblock(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t first) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.eq.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %3, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %3, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %3, 1;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(first), "r"(a_tmem + 8), "l"(b_desc + 2),
      "r"(a_tmem + 16), "l"(b_desc + 4), "r"(a_tmem + 24), "l"(b_desc + 6)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Warp-wide: thread i writes 16 consecutive 32-bit columns of lane
// (lane field of taddr) + i.
__device__ __forceinline__ void tmem_st_16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

// Warp-wide: thread i reads 16 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_ld_16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row groups 1024 bytes apart), as
// written by a TMA load with CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte
// aligned buffer.
__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFF);   // start address
  d |= static_cast<uint64_t>(1) << 16;                      // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;              // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                      // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B of the same
// 16-bit type (0 = f16, 1 = bf16), both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t ab_type, uint32_t M, uint32_t N) {
  return (1u << 4)                // D format: f32
         | (ab_type << 7)         // A format
         | (ab_type << 10)        // B format
         | ((N >> 3) << 17)       // N / 8
         | ((M >> 4) << 24);      // M / 16
}

}  // namespace tmw4

// api.cu -- the C ABI of libtmw4 (declared in include/tmw4.h): argument
// validation, the packed-weight handle, the per-device error word, the
// per-(device, stream) split-K workspace, TMA descriptor creation, variant
// selection and the measured-throughput tuner.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "kernels.h"
#include "tmw4.h"
#include "tmw4_device.cuh"

using namespace tmw4;

// ----------------------------------------------------------------- handle
static constexpr uint32_t kPackedMagic = 0x34574D54u;  // "TMW4"

struct tm_packed {
  uint32_t magic;
  int K, N, group;
  tm_dtype dtype;
  int symmetric;
  int bits;   // 4, or 8
  int fp8;    // 8-bit codes are FP8 E4M3
  int device;
  uint8_t *qw;
  uint16_t *scales;
  uint8_t *zeros;
  size_t qw_bytes, scales_bytes, zeros_bytes;
};

// ------------------------------------------------------------ last error
static thread_local std::string g_last_error;

static tm_status fail(tm_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

static tm_status fail_cuda(cudaError_t e, const char *what) {
  return fail(e == cudaErrorMemoryAllocation ? TM_ERR_OOM : TM_ERR_CUDA, "%s: %s (%s)", what,
              cudaGetErrorName(e), cudaGetErrorString(e));
}

#define TM_CUDA(call, what)                      \
  do {                                           \
    cudaError_t _e = (call);                     \
    if (_e != cudaSuccess) return fail_cuda(_e, what); \
  } while (0)

// Bounded waits give up after this long (nanoseconds); TM_WAIT_LIMIT_NS
// overrides it.  No legitimate wait comes near it.
static unsigned long long wait_limit_ns() {
  static unsigned long long v = [] {
    const char *e = getenv("TM_WAIT_LIMIT_NS");
    unsigned long long x = e ? strtoull(e, nullptr, 10) : 0ull;
    return (x >= 1000ull && x <= 60000000000ull) ? x : 4000000000ull;
  }();
  return v;
}

// GEMM launches overlap the previous kernel in the stream (programmatic
// dependent launch) unless TM_PDL=0.
static bool pdl_enabled() {
  static const bool v = [] {
    const char *e = getenv("TM_PDL");
    return !(e != nullptr && e[0] == '0' && e[1] == '\0');
  }();
  return v;
}

// --------------------------------------------------- per-device state
static std::mutex g_mu;
static constexpr int kMaxDevices = 64;
static unsigned int *g_err_word[kMaxDevices] = {};

static tm_status current_device(int *dev) {
  TM_CUDA(cudaGetDevice(dev), "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return fail(TM_ERR_UNSUPPORTED, "device index %d", *dev);
  return TM_OK;
}

static tm_status error_word(int dev, unsigned int **out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_word[dev] == nullptr) {
    unsigned int *p = nullptr;
    TM_CUDA(cudaMalloc(&p, TM_ERR_WORDS * sizeof(unsigned int)), "cudaMalloc(error word)");
    TM_CUDA(cudaMemset(p, 0, TM_ERR_WORDS * sizeof(unsigned int)), "cudaMemset(error word)");
    g_err_word[dev] = p;
  }
  *out = g_err_word[dev];
  return TM_OK;
}

struct Workspace {
  float *ws = nullptr;
  size_t ws_bytes = 0;
  unsigned int *counters = nullptr;
  size_t n_counters = 0;
};
static std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

static bool stream_capturing(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return false;
  return cs != cudaStreamCaptureStatusNone;
}

// Workspace of (dev, st) with at least the given sizes; grows outside capture.
static tm_status get_workspace(int dev, cudaStream_t st, size_t ws_bytes, size_t n_counters,
                               Workspace **out) {
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace &w = g_ws[{dev, st}];
  if (w.ws_bytes < ws_bytes || w.n_counters < n_counters) {
    if (stream_capturing(st))
      return fail(TM_ERR_UNSUPPORTED,
                  "split-K workspace must grow (%zu B) while the stream is being captured; "
                  "run this shape once outside capture first",
                  ws_bytes);
    // the old buffers may still be in use by queued work on this stream
    TM_CUDA(cudaStreamSynchronize(st), "cudaStreamSynchronize");
    if (w.ws_bytes < ws_bytes) {
      if (w.ws) cudaFree(w.ws);
      w.ws = nullptr;
      w.ws_bytes = 0;
      size_t sz = std::max(ws_bytes, static_cast<size_t>(1) << 20);
      TM_CUDA(cudaMalloc(&w.ws, sz), "cudaMalloc(split-K workspace)");
      w.ws_bytes = sz;
    }
    if (w.n_counters < n_counters) {
      if (w.counters) cudaFree(w.counters);
      w.counters = nullptr;
      w.n_counters = 0;
      size_t n = std::max(n_counters, static_cast<size_t>(4096));
      TM_CUDA(cudaMalloc(&w.counters, n * sizeof(unsigned int)), "cudaMalloc(counters)");
      TM_CUDA(cudaMemsetAsync(w.counters, 0, n * sizeof(unsigned int), st), "cudaMemsetAsync");
      TM_CUDA(cudaStreamSynchronize(st), "cudaStreamSynchronize");
      w.n_counters = n;
    }
  }
  *out = &w;
  return TM_OK;
}

// ------------------------------------------------------------ TMA encode
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static tm_status get_encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr)
      return fail(TM_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *fn = g_encode;
  return TM_OK;
}

// Activation tensor map with the 128-byte swizzle; rows past M read as
// zero.  Preferred form: 3-D (64 x M x K/64, strides K*2 and 128 bytes) so
// that one copy brings `kbs` consecutive 64-K blocks of BLOCK_M rows, each
// block landing as its own swizzled [block_m][64] tile.  If the driver
// rejects that map, a 2-D map (box 64 x block_m, one copy per 64-K block)
// is used instead and *is_3d is 0.
static int g_map3d_ok = -1;   // -1 unknown, 0 rejected, 1 accepted

static tm_status encode_act_map(const void *A, int M, int K, bool bf16, int block_m, int kbs,
                                CUtensorMap *map, int *is_3d) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  tm_status s = get_encoder(&enc);
  if (s != TM_OK) return s;
  const CUtensorMapDataType dt =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint32_t estr[3] = {1, 1, 1};
  if (g_map3d_ok != 0) {
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(block_m), static_cast<cuuint32_t>(kbs)};
    CUresult r = enc(map, dt, 3, const_cast<void *>(A), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
      g_map3d_ok = 1;
      *is_3d = 1;
      return TM_OK;
    }
    g_map3d_ok = 0;
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(block_m)};
  CUresult r = enc(map, dt, 2, const_cast<void *>(A), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  *is_3d = 0;
  return TM_OK;
}

// ------------------------------------------------------------ validation
static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static tm_status check_handle(const tm_packed *W) {
  if (W == nullptr) return fail(TM_ERR_INVALID_ARG, "packed weight handle is NULL");
  if (W->magic != kPackedMagic) return fail(TM_ERR_INVALID_ARG, "not a packed weight handle");
  return TM_OK;
}

// -------------------------------------------------------- variant choice
// The selection table is keyed by shape, format and row-count bucket: the
// next power of two >= M (every kernel's row limits are powers of two, so
// one bucket has one set of legal variants).
static int m_bucket(int M) {
  int b = 1;
  while (b < M && b < (1 << 30)) b <<= 1;
  return b;
}
// fmt: code format, 0 int4, 1 int8, 2 FP8
struct TuneKey {
  int N, K, group, dtype, sym, mb, fmt;
  bool operator<(const TuneKey &o) const {
    return std::tie(N, K, group, dtype, sym, mb, fmt) < std::tie(o.N, o.K, o.group, o.dtype, o.sym, o.mb, o.fmt);
  }
};
static int code_format(const tm_packed *W) { return W->bits == 8 ? (W->fp8 ? 2 : 1) : 0; }
static TuneKey tune_key(const tm_packed *W, int M) {
  return TuneKey{W->N, W->K, W->group, (int)W->dtype, W->symmetric, m_bucket(M), code_format(W)};
}
struct TuneVal {
  tm_config cfg;
  double us;
  int M;   // the row count that was measured
};
static std::map<TuneKey, TuneVal> g_tune;

static int sm_count(int dev) {
  static std::atomic<int> cached[kMaxDevices] = {};
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

static int gemv_rows_tmpl(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

// Is cfg runnable for this shape?  (Fills defaults for zero fields.)
static bool normalize_config(const tm_packed *W, int M, tm_config *c, std::string *why) {
  const int KB = W->K / 64;
  // Groups of 32 need a second scale inside each 64-K block: the kernels
  // that scale the dequantized weight before the multiply (TC, CUDA-core
  // GEMV) take them; those that scale fp32 sums per block do not.
  if (W->group == 32 && (c->kernel == TM_KERNEL_DECODE_MMA || c->kernel == TM_KERNEL_TC_DECODE ||
                         (c->kernel == TM_KERNEL_GEMV && c->dq_warps == 1))) {
    if (why) *why = "this kernel needs groups of at least 64";
    return false;
  }
  // 8-bit codes run on the CUDA-core GEMV, the register-MMA decode kernel
  // (up to two K-groups) and the TC kernel
  if (W->bits == 8 && !(c->kernel == TM_KERNEL_TC || (c->kernel == TM_KERNEL_GEMV && c->dq_warps == 0) ||
                        (c->kernel == TM_KERNEL_DECODE_MMA && c->dq_warps != 16))) {
    if (why) *why = "8-bit weights run on the CUDA-core GEMV, DECODE_MMA (dq_warps up to 8) and the TC kernel";
    return false;
  }
  if (c->kernel == TM_KERNEL_DECODE_MMA) {
    if (decode_mma_nt8(M) == 0) {
      if (why) *why = "DECODE_MMA handles M <= 16";
      return false;
    }
    c->block_m = 8 * decode_mma_nt8(M);
    if (c->dq_warps == 1 || c->dq_warps == 2) {
      // cluster split-K with dq_warps K-groups of four consumer warps:
      // split_k = CTAs per cluster, normalized to the group-aligned split
      // that covers K
      int per = 0;
      const int S = decode_mma_cluster_split(W->dtype == TM_BF16, M, W->K, W->group, c->dq_warps,
                                             c->split_k <= 0 ? 1 : c->split_k, &per, W->bits);
      if (S == 0) {
        if (why) *why = "DECODE_MMA cluster of that size cannot be resident";
        return false;
      }
      c->split_k = S;
      return true;
    }
    // stream-K: dq_warps = consumer warps per CTA (4, 8 or 16; 0 = 4),
    // split_k = persistent CTAs per SM (clamped to what fits; 0 = all that fit)
    if (c->dq_warps == 0) c->dq_warps = 4;
    if (c->dq_warps != 4 && c->dq_warps != 8 && c->dq_warps != 16) {
      if (why) *why = "DECODE_MMA takes dq_warps 4, 8 or 16 (stream-K) or 1, 2 (clusters)";
      return false;
    }
    const int occ = decode_mma_ctas_per_sm(W->dtype == TM_BF16, M, W->group, c->dq_warps / 4, W->bits);
    if (c->split_k <= 0 || c->split_k > occ) c->split_k = occ;
    return true;
  }
  if (c->split_k <= 0) c->split_k = 1;
  if (c->split_k > KB) {
    if (why) *why = "split_k larger than K/64";
    return false;
  }
  if (c->kernel == TM_KERNEL_GEMV) {
    // dq_warps: 0 = CUDA-core FMAs (M <= 8), 1 = tensor-core MMAs (M <= 16)
    if (c->dq_warps != 0 && c->dq_warps != 1) {
      if (why) *why = "GEMV takes dq_warps 0 (CUDA cores) or 1 (tensor cores)";
      return false;
    }
    const bool mma = c->dq_warps == 1;
    if (M > (mma ? 16 : 8)) {
      if (why) *why = mma ? "GEMV with tensor cores handles M <= 16" : "GEMV handles M <= 8";
      return false;
    }
    const int kb_per = (KB + c->split_k - 1) / c->split_k;
    const int rows = mma ? (M <= 8 ? 8 : 16) : gemv_rows_tmpl(M);
    const size_t smem = mma ? gemv_mma_smem_bytes(rows / 8, kb_per, W->group) : gemv_smem_bytes(rows, kb_per);
    if (smem > 200 * 1024) {
      if (why) *why = "GEMV K range too long for shared memory; raise split_k";
      return false;
    }
    c->block_m = rows;
    return true;
  }
  if (c->kernel == TM_KERNEL_TC) {
    if (c->block_m != 16 && c->block_m != 32 && c->block_m != 64 && c->block_m != 128 &&
        c->block_m != 256) {
      if (why) *why = "TC block_m must be 16, 32, 64, 128 or 256";
      return false;
    }
    if (c->dq_warps == 0) c->dq_warps = 8;
    if (c->dq_warps != 4 && c->dq_warps != 8 && c->dq_warps != 16) {
      if (why) *why = "TC dq_warps must be 4, 8 or 16";
      return false;
    }
    if (!tc_variant_ok(c->block_m, c->dq_warps, W->bits)) {
      if (why) *why = "this block_m has too few pipeline stages for that many dequant warps";
      return false;
    }
    if ((M + c->block_m - 1) / c->block_m > 65535) {
      if (why) *why = "too many row tiles";
      return false;
    }
    return true;
  }
  if (c->kernel == TM_KERNEL_TC_DECODE) {
    if (c->block_m != 16 && c->block_m != 32 && c->block_m != 64) {
      if (why) *why = "TC_DECODE block_m must be 16, 32 or 64";
      return false;
    }
    if (c->dq_warps == 0) c->dq_warps = 8;
    if (!tc_decode_ok(c->block_m, c->dq_warps)) {
      if (why) *why = "TC_DECODE dq_warps must be 4, 8, 12 or 16 (12 and 16 only with block_m <= 32)";
      return false;
    }
    c->split_k = 1;   // stream-K: the grid divides the work itself
    if ((M + c->block_m - 1) / c->block_m > 65535) {
      if (why) *why = "too many row tiles";
      return false;
    }
    return true;
  }
  if (why) *why = "unknown kernel family";
  return false;
}

// Built-in rule used when the tuned table has no entry for this shape, from
// the crossovers measured on GB300: the CUDA-core GEMV for one or two rows
// (about three CTAs per SM over K splits), the tcgen05 decode kernel up to 64
// rows, the tcgen05 kernel beyond.  The register-MMA decode kernel is picked
// by the tuner where it measures faster.
static tm_config default_config(const tm_packed *W, int M, int dev) {
  const int KB = W->K / 64;
  const int sms = sm_count(dev);
  tm_config c{};
  std::string why;
  // Measured on GB300 (graphs of back-to-back launches over weights larger
  // than L2): up to 4 rows, weights of at most 16 MB run fastest in clusters
  // of 8 CTAs per tile (no split-K workspace round trip); otherwise up to 8
  // rows the persistent stream-K grid of the register-MMA kernel; beyond,
  // the tcgen05 decode kernel up to 64 rows and the tcgen05 kernel after.
  const double wbytes = static_cast<double>(W->N) * W->K / 2;
  if ((W->group == 32 || W->bits == 8) && M <= 8) {
    c = tm_config{TM_KERNEL_GEMV, 0, 4, 0};
    while (!normalize_config(W, M, &c, &why) && c.split_k < KB) c.split_k = std::min(KB, c.split_k * 2);
    if (normalize_config(W, M, &c, &why)) return c;
  }
  if (M <= 4 && wbytes <= 16e6) {
    c = tm_config{TM_KERNEL_DECODE_MMA, 0, 8, 1};
    if (normalize_config(W, M, &c, &why)) return c;
  }
  if (M <= 8) {
    c = tm_config{TM_KERNEL_DECODE_MMA, 0, 0, 4};
    if (normalize_config(W, M, &c, &why)) return c;
  }
  if (W->bits == 8 && M <= 16) {
    c = tm_config{TM_KERNEL_DECODE_MMA, 0, 0, 4};
    if (normalize_config(W, M, &c, &why)) return c;
  }
  if (M <= 64) {
    c = tm_config{TM_KERNEL_TC_DECODE, M <= 16 ? 16 : M <= 32 ? 32 : 64, 1, 8};
    if (normalize_config(W, M, &c, &why)) return c;
  }
  c = tm_config{};
  c.kernel = TM_KERNEL_TC;
  c.block_m = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  c.dq_warps = 8;
  const int per_sm = c.block_m <= 64 ? 2 : 1;
  const int tiles = (W->N / 128) * ((M + c.block_m - 1) / c.block_m);
  int s = 1;
  if (tiles < sms * per_sm) {
    s = (sms * per_sm + tiles - 1) / tiles;
    s = std::min(s, std::max(1, KB / 4));
    s = std::min(s, 32);
  }
  c.split_k = s;
  normalize_config(W, M, &c, &why);
  return c;
}

static void load_tune_env_once();

// TM_VARIANT="kernel:block_m:split_k:dq_warps" (kernel by name -- gemv, tc,
// tc_decode, decode_mma -- or number) forces one variant for every GEMM it
// can run; shapes it cannot run keep the regular selection.
struct VariantOverride {
  bool set = false;
  tm_config cfg{};
};
static const VariantOverride &variant_override() {
  static const VariantOverride v = [] {
    VariantOverride o;
    const char *e = getenv("TM_VARIANT");
    if (e == nullptr || *e == 0) return o;
    char name[32] = {};
    int bm = 0, sk = 1, dq = 0;
    if (sscanf(e, "%31[^:]:%d:%d:%d", name, &bm, &sk, &dq) < 1) return o;
    int k = atoi(name);
    if (strcmp(name, "gemv") == 0) k = TM_KERNEL_GEMV;
    else if (strcmp(name, "tc") == 0) k = TM_KERNEL_TC;
    else if (strcmp(name, "tc_decode") == 0) k = TM_KERNEL_TC_DECODE;
    else if (strcmp(name, "decode_mma") == 0) k = TM_KERNEL_DECODE_MMA;
    if (k < TM_KERNEL_GEMV || k > TM_KERNEL_DECODE_MMA) return o;
    o.set = true;
    o.cfg = tm_config{k, bm, sk, dq};
    return o;
  }();
  return v;
}

static tm_config select_config(const tm_packed *W, int M, int dev) {
  const VariantOverride &ov = variant_override();
  if (ov.set) {
    tm_config c = ov.cfg;
    if (normalize_config(W, M, &c, nullptr)) return c;
  }
  load_tune_env_once();
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_tune.find(tune_key(W, M));
    if (it != g_tune.end()) {
      tm_config c = it->second.cfg;
      if (normalize_config(W, M, &c, nullptr)) return c;
    }
  }
  return default_config(W, M, dev);
}

// Launched (plainly) after the kernels of a repack.  A GEMM that follows on
// the same stream is launched with programmatic dependent launch and reads
// its packed weights before griddepcontrol.wait, so it may overlap the
// kernel just before it; with this empty kernel in between, that kernel is
// never the repack, whose writes are complete and visible by plain stream
// order before this one starts.
static __global__ void pack_fence_kernel() {}

#ifdef TMW4_TRACE
// debug builds only: device buffer that receives the per-stage cycle stamps
static long long *g_trace = nullptr;
extern "C" tm_status tm_debug_set_trace(void *p) {
  g_trace = static_cast<long long *>(p);
  return TM_OK;
}
static __global__ void debug_marker_kernel(long long *out, int idx) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  if (threadIdx.x == 0) out[idx] = static_cast<long long>(t);
}
// debug builds only: a one-thread kernel that records %globaltimer at out[idx]
extern "C" tm_status tm_debug_marker(void *out, int idx, void *stream) {
  debug_marker_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<long long *>(out), idx);
  return cudaGetLastError() == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}
#endif

// ------------------------------------------------------------ GEMM launch
// K split and scratch of a launch: GEMV and TC split K evenly (TC on stage
// boundaries; trailing splits that would be empty are dropped); TC_DECODE
// divides (tile, stage) units over a persistent grid and needs partial slots
// only where the grid cuts a tile.
static void plan_work(const tm_packed *W, int M, const tm_config &cfg, GemmArgs *a, int *dec_grid,
                      size_t *ws_floats, size_t *n_counters) {
  const int KB = W->K / 64;
  *ws_floats = 0;
  *n_counters = 0;
  if (cfg.kernel == TM_KERNEL_DECODE_MMA && (cfg.dq_warps == 1 || cfg.dq_warps == 2)) {
    int per = KB;
    a->splits = decode_mma_cluster_split(W->dtype == TM_BF16, M, W->K, W->group, cfg.dq_warps, cfg.split_k, &per,
                                         W->bits);
    a->kb_per_split = per;
    a->ws_slots = 1;
    *dec_grid = W->N / 128;
    return;
  }
  if (cfg.kernel == TM_KERNEL_DECODE_MMA) {
    long long tiles = 0;
    int slots = 1;
    decode_mma_plan(M, W->N, W->K, W->group, cfg.split_k * sm_count(W->device), dec_grid, &tiles,
                    &slots);
    a->kb_per_split = KB;
    a->splits = 1;
    a->ws_slots = slots;
    if (slots > 1) {
      *ws_floats = static_cast<size_t>(tiles) * slots * M * 128;
      *n_counters = static_cast<size_t>(tiles);
    }
    return;
  }
  if (cfg.kernel == TM_KERNEL_TC_DECODE) {
    long long tiles = 0;
    int slots = 1;
    tc_decode_plan(M, W->N, W->K, cfg.block_m, sm_count(W->device), dec_grid, &tiles, &slots);
    a->kb_per_split = KB;
    a->splits = 1;
    a->ws_slots = slots;
    if (slots > 1) {
      *ws_floats = static_cast<size_t>(tiles) * slots * 128 * cfg.block_m;
      *n_counters = static_cast<size_t>(tiles);
    }
    return;
  }
  const int gran = cfg.kernel == TM_KERNEL_TC ? tc_kblocks_per_stage(cfg.block_m) : 1;
  int per = (KB + cfg.split_k - 1) / cfg.split_k;
  per = (per + gran - 1) / gran * gran;
  a->kb_per_split = per;
  a->splits = (KB + per - 1) / per;
  if (a->splits > 1) {
    *ws_floats = static_cast<size_t>(a->splits) * M * W->N;
    *n_counters = cfg.kernel == TM_KERNEL_GEMV
                      ? static_cast<size_t>(W->N / 64)
                      : static_cast<size_t>(W->N / 128) * ((M + cfg.block_m - 1) / cfg.block_m);
  }
}

// Launches the planned variant (arguments, workspace and grid already set).
static tm_status launch_planned(const void *A, const tm_packed *W, int M, const tm_config &cfg,
                                GemmArgs &a, int dec_grid, cudaStream_t st, const char *what) {
  const bool bf16 = W->dtype == TM_BF16;
  cudaError_t e;
  if (cfg.kernel == TM_KERNEL_GEMV) {
    e = launch_gemv(a, bf16, cfg.block_m, cfg.dq_warps == 1, st);
  } else if (cfg.kernel == TM_KERNEL_DECODE_MMA) {
    CUtensorMap map;
    tm_status s = encode_act_map(A, M, W->K, bf16, cfg.block_m, 1, &map, &a.act_map_3d);
    if (s != TM_OK) return s;
    e = cfg.dq_warps <= 2 ? launch_decode_mma(a, map, bf16, cfg.dq_warps, dec_grid, a.splits, st)
                          : launch_decode_mma(a, map, bf16, cfg.dq_warps / 4, dec_grid, 0, st);
  } else if (cfg.kernel == TM_KERNEL_TC_DECODE) {
    CUtensorMap map;
    tm_status s = encode_act_map(A, M, W->K, bf16, cfg.block_m, tc_decode_kblocks_per_stage(), &map,
                                 &a.act_map_3d);
    if (s != TM_OK) return s;
    e = launch_tc_decode(a, map, bf16, cfg.block_m, cfg.dq_warps, dec_grid, st);
  } else {
    CUtensorMap map;
    tm_status s = encode_act_map(A, M, W->K, bf16, cfg.block_m, tc_kblocks_per_stage(cfg.block_m),
                                 &map, &a.act_map_3d);
    if (s != TM_OK) return s;
    e = launch_tc(a, map, bf16, cfg.block_m, cfg.dq_warps, st);
  }
  if (e != cudaSuccess) return fail_cuda(e, what);
  return TM_OK;
}

static tm_status run_gemm(const void *A, const tm_packed *W, void *C, int M, const tm_config &cfg,
                          cudaStream_t st) {
  unsigned int *err = nullptr;
  tm_status s = error_word(W->device, &err);
  if (s != TM_OK) return s;
  GemmArgs a{};
  a.qw = W->qw;
  a.scales = W->scales;
  a.zeros = W->symmetric ? nullptr : W->zeros;
  a.A = static_cast<const uint16_t *>(A);
  a.C = static_cast<uint16_t *>(C);
  a.err = err;
  a.M = M;
  a.N = W->N;
  a.K = W->K;
  a.group = W->group;
  a.wbits = W->bits;
  a.fp8 = W->fp8;
  int dec_grid = 0;
  size_t ws_floats = 0, n_counters = 0;
  plan_work(W, M, cfg, &a, &dec_grid, &ws_floats, &n_counters);
  a.limit_ns = wait_limit_ns();
  a.pdl = pdl_enabled() ? 1 : 0;
#ifdef TMW4_TRACE
  a.trace = g_trace;
#endif
  if (ws_floats > 0) {
    Workspace *ws = nullptr;
    s = get_workspace(W->device, st, sizeof(float) * ws_floats, n_counters, &ws);
    if (s != TM_OK) return s;
    a.ws = ws->ws;
    a.counters = ws->counters;
  }
  return launch_planned(A, W, M, cfg, a, dec_grid, st, "kernel launch");
}

static tm_status check_gemm_args(const void *A, const tm_packed *W, const void *C, int M, int N,
                                 int K) {
  tm_status s = check_handle(W);
  if (s != TM_OK) return s;
  if (N != W->N || K != W->K)
    return fail(TM_ERR_INVALID_ARG, "shape (N=%d, K=%d) does not match the packed weight (N=%d, K=%d)",
                N, K, W->N, W->K);
  if (M < 0) return fail(TM_ERR_INVALID_ARG, "M must be >= 0");
  if (M > 65535 * 256) return fail(TM_ERR_UNSUPPORTED, "M too large");
  if (M == 0) return TM_OK;
  if (A == nullptr || C == nullptr) return fail(TM_ERR_INVALID_ARG, "A and C must not be NULL");
  if (!aligned16(A) || !aligned16(C))
    return fail(TM_ERR_INVALID_ARG, "A and C must be 16-byte aligned");
  int dev = -1;
  s = current_device(&dev);
  if (s != TM_OK) return s;
  if (dev != W->device)
    return fail(TM_ERR_INVALID_ARG, "packed weight lives on device %d, current device is %d",
                W->device, dev);
  return TM_OK;
}

// Reads and clears the static error word of tm_gemm_w4a16_noalloc on device
// `dev` (zeros if that entry point has not run on the device yet).
static tm_status take_static_error(int dev, unsigned int (&w)[TM_ERR_WORDS]);

// ================================================================ C ABI
extern "C" tm_status tm_tc_decode_pipeline(int block_m, int dq_warps, int *weight_stages,
                                           int *act_stages_per_wg, int *tmem_slots_per_wg,
                                           int *legal) {
  if (weight_stages == nullptr || act_stages_per_wg == nullptr || tmem_slots_per_wg == nullptr ||
      legal == nullptr)
    return fail(TM_ERR_INVALID_ARG, "output pointers must not be NULL");
  *legal = tc_decode_ok(block_m, dq_warps) ? 1 : 0;
  if (block_m != 16 && block_m != 32 && block_m != 64)
    return fail(TM_ERR_INVALID_ARG, "block_m must be 16, 32 or 64");
  if (dq_warps != 4 && dq_warps != 8 && dq_warps != 12 && dq_warps != 16)
    return fail(TM_ERR_INVALID_ARG, "dq_warps must be 4, 8, 12 or 16");
  tc_decode_pipeline(block_m, dq_warps, weight_stages, act_stages_per_wg, tmem_slots_per_wg);
  return TM_OK;
}

extern "C" tm_status tm_decode_plan(int M, int N, int K, int block_m, int sm_count, int *grid,
                                    long long *tiles, int *partial_slots) {
  if (grid == nullptr || tiles == nullptr || partial_slots == nullptr)
    return fail(TM_ERR_INVALID_ARG, "output pointers must not be NULL");
  if (M <= 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 64 != 0 || sm_count <= 0)
    return fail(TM_ERR_INVALID_ARG, "need M, N, K, sm_count > 0, N %% 128 == 0, K %% 64 == 0");
  if (block_m != 16 && block_m != 32 && block_m != 64)
    return fail(TM_ERR_INVALID_ARG, "block_m must be 16, 32 or 64");
  tc_decode_plan(M, N, K, block_m, sm_count, grid, tiles, partial_slots);
  return TM_OK;
}

extern "C" {

const char *tm_version(void) { return "tmw4 0.1 (sm_103a)"; }

const char *tm_last_error(void) { return g_last_error.c_str(); }

// The group the kernels run with for a source group G: 32, 64 or 128.  A
// coarser group (any multiple of 64, per-channel G = K included) is packed
// as 128 when it is a multiple of 128, else as 64, each of its scales and
// zeros repeated over the finer groups it spans: the dequantized weight is
// identical by construction.
static int packed_group(int group) { return group == 32 ? 32 : group % 128 == 0 ? 128 : 64; }

// Packs codes in layout `src` (q: u8 [K][N], AWQ int32 [K][N/8] or GPTQ
// int32 [K/8][N]), fp16/bf16 scales [K/G][N] and zeros (same layout family
// as q: u8 [K/G][N] or int32 [K/G][N/8]; NULL = symmetric, z = 8).
static tm_status pack_common(int src, const void *q, const void *scales, const void *zeros, int zero_offset,
                             int K, int N, int group, tm_dtype dtype, void *stream, tm_packed **out,
                             const char *what) {
  if (out == nullptr) return fail(TM_ERR_INVALID_ARG, "out must not be NULL");
  *out = nullptr;
  if (q == nullptr || scales == nullptr) return fail(TM_ERR_INVALID_ARG, "codes and scales must not be NULL");
  if (dtype != TM_F16 && dtype != TM_BF16) return fail(TM_ERR_INVALID_ARG, "dtype must be TM_F16 or TM_BF16");
  if (K <= 0 || N <= 0) return fail(TM_ERR_INVALID_ARG, "K and N must be positive");
  if (group != 32 && (group <= 0 || group % 64 != 0))
    return fail(TM_ERR_INVALID_ARG, "group must be 32 or a positive multiple of 64");
  if (K % group != 0 || K % 64 != 0)
    return fail(TM_ERR_INVALID_ARG, "K (%d) must be a multiple of group (%d) and of 64", K, group);
  if (N % 128 != 0) return fail(TM_ERR_INVALID_ARG, "N (%d) must be a multiple of 128", N);
  if (!aligned16(q) || !aligned16(scales) || (zeros && !aligned16(zeros)))
    return fail(TM_ERR_INVALID_ARG, "codes, scales and zeros must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = -1;
  tm_status s = current_device(&dev);
  if (s != TM_OK) return s;
  unsigned int *err = nullptr;
  s = error_word(dev, &err);
  if (s != TM_OK) return s;
  const int G = packed_group(group), rep = group / G;

  tm_packed *W = new tm_packed{};
  W->magic = kPackedMagic;
  W->K = K;
  W->N = N;
  W->group = G;
  W->dtype = dtype;
  W->symmetric = zeros == nullptr ? 1 : 0;
  W->bits = 4;
  W->fp8 = 0;
  W->device = dev;
  W->qw_bytes = static_cast<size_t>(K) * N / 2;
  W->scales_bytes = static_cast<size_t>(K / G) * N * 2;
  W->zeros_bytes = zeros ? static_cast<size_t>(K / G) * (N / 2) : 0;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&W->qw), W->qw_bytes, st);
  if (e == cudaSuccess) e = cudaMallocAsync(reinterpret_cast<void **>(&W->scales), W->scales_bytes, st);
  if (e == cudaSuccess && zeros)
    e = cudaMallocAsync(reinterpret_cast<void **>(&W->zeros), W->zeros_bytes, st);
  if (e == cudaSuccess) e = launch_repack(q, W->qw, K, N, src, err, st);
  if (e == cudaSuccess)
    e = launch_pack_scales(static_cast<const uint16_t *>(scales), W->scales, K / G, N, rep, st);
  if (e == cudaSuccess && zeros) e = launch_pack_zeros(zeros, W->zeros, K / G, N, rep, src, zero_offset, err, st);
  if (e == cudaSuccess) {
    pack_fence_kernel<<<1, 1, 0, st>>>();
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    if (W->qw) cudaFreeAsync(W->qw, st);
    if (W->scales) cudaFreeAsync(W->scales, st);
    if (W->zeros) cudaFreeAsync(W->zeros, st);
    W->magic = 0;
    delete W;
    return fail_cuda(e, what);
  }
  *out = W;
  return TM_OK;
}

tm_status tm_pack_w4(const uint8_t *q, const void *scales, const uint8_t *zeros, int K, int N,
                     int group, tm_dtype dtype, void *stream, tm_packed **out) {
  return pack_common(SRC_U8, q, scales, zeros, 0, K, N, group, dtype, stream, out, "tm_pack_w4");
}

tm_status tm_pack_awq(const int32_t *qweight, const int32_t *qzeros, const void *scales, int K, int N,
                      int group, tm_dtype dtype, void *stream, tm_packed **out) {
  return pack_common(SRC_AWQ, qweight, scales, qzeros, 0, K, N, group, dtype, stream, out, "tm_pack_awq");
}

tm_status tm_pack_gptq(const int32_t *qweight, const int32_t *qzeros, const void *scales, int zero_offset,
                       int K, int N, int group, tm_dtype dtype, void *stream, tm_packed **out) {
  if (zero_offset != 0 && zero_offset != 1) return fail(TM_ERR_INVALID_ARG, "zero_offset must be 0 or 1");
  if (K % 8 != 0) return fail(TM_ERR_INVALID_ARG, "K must be a multiple of 8");
  return pack_common(SRC_GPTQ, qweight, scales, qzeros, zero_offset, K, N, group, dtype, stream, out,
                     "tm_pack_gptq");
}

// Packs 8-bit codes (u8 [K][N]): int8 with byte zeros [K/G][N] (NULL:
// symmetric, zero 128), or FP8 E4M3 (fp8 = 1, no zeros).
static tm_status pack8_common(const uint8_t *q, const void *scales, const uint8_t *zeros, int fp8, int K, int N,
                              int group, tm_dtype dtype, void *stream, tm_packed **out, const char *what) {
  if (out == nullptr) return fail(TM_ERR_INVALID_ARG, "out must not be NULL");
  *out = nullptr;
  if (q == nullptr || scales == nullptr) return fail(TM_ERR_INVALID_ARG, "codes and scales must not be NULL");
  if (dtype != TM_F16 && dtype != TM_BF16) return fail(TM_ERR_INVALID_ARG, "dtype must be TM_F16 or TM_BF16");
  if (K <= 0 || N <= 0) return fail(TM_ERR_INVALID_ARG, "K and N must be positive");
  if (group != 32 && (group <= 0 || group % 64 != 0))
    return fail(TM_ERR_INVALID_ARG, "group must be 32 or a positive multiple of 64");
  if (K % group != 0 || K % 64 != 0)
    return fail(TM_ERR_INVALID_ARG, "K (%d) must be a multiple of group (%d) and of 64", K, group);
  if (N % 128 != 0) return fail(TM_ERR_INVALID_ARG, "N (%d) must be a multiple of 128", N);
  if (!aligned16(q) || !aligned16(scales) || (zeros && !aligned16(zeros)))
    return fail(TM_ERR_INVALID_ARG, "codes, scales and zeros must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = -1;
  tm_status s = current_device(&dev);
  if (s != TM_OK) return s;
  const int G = packed_group(group), rep = group / G;
  tm_packed *W = new tm_packed{};
  W->magic = kPackedMagic;
  W->K = K;
  W->N = N;
  W->group = G;
  W->dtype = dtype;
  W->symmetric = zeros == nullptr ? 1 : 0;
  W->bits = 8;
  W->fp8 = fp8;
  W->device = dev;
  W->qw_bytes = static_cast<size_t>(K) * N;
  W->scales_bytes = static_cast<size_t>(K / G) * N * 2;
  W->zeros_bytes = zeros ? static_cast<size_t>(K / G) * N : 0;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&W->qw), W->qw_bytes, st);
  if (e == cudaSuccess) e = cudaMallocAsync(reinterpret_cast<void **>(&W->scales), W->scales_bytes, st);
  if (e == cudaSuccess && zeros) e = cudaMallocAsync(reinterpret_cast<void **>(&W->zeros), W->zeros_bytes, st);
  if (e == cudaSuccess) e = launch_repack8(q, W->qw, K, N, st);
  if (e == cudaSuccess)
    e = launch_pack_scales(static_cast<const uint16_t *>(scales), W->scales, K / G, N, rep, st);
  if (e == cudaSuccess && zeros) e = launch_pack_zeros8(zeros, W->zeros, K / G, N, rep, st);
  if (e == cudaSuccess) {
    pack_fence_kernel<<<1, 1, 0, st>>>();
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    if (W->qw) cudaFreeAsync(W->qw, st);
    if (W->scales) cudaFreeAsync(W->scales, st);
    if (W->zeros) cudaFreeAsync(W->zeros, st);
    W->magic = 0;
    delete W;
    return fail_cuda(e, what);
  }
  *out = W;
  return TM_OK;
}

tm_status tm_pack_w8(const uint8_t *q, const void *scales, const uint8_t *zeros, int K, int N, int group,
                     tm_dtype dtype, void *stream, tm_packed **out) {
  return pack8_common(q, scales, zeros, 0, K, N, group, dtype, stream, out, "tm_pack_w8");
}

tm_status tm_pack_fp8(const uint8_t *q, const void *scales, int K, int N, int group, tm_dtype dtype,
                      void *stream, tm_packed **out) {
  return pack8_common(q, scales, nullptr, 1, K, N, group, dtype, stream, out, "tm_pack_fp8");
}

tm_status tm_packed_free(tm_packed *W, void *stream) {
  if (W == nullptr) return TM_OK;
  tm_status s = check_handle(W);
  if (s != TM_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (W->qw) cudaFreeAsync(W->qw, st);
  if (W->scales) cudaFreeAsync(W->scales, st);
  if (W->zeros) cudaFreeAsync(W->zeros, st);
  W->magic = 0;
  delete W;
  return TM_OK;
}

tm_status tm_packed_get(const tm_packed *W, tm_packed_info *info) {
  tm_status s = check_handle(W);
  if (s != TM_OK) return s;
  if (info == nullptr) return fail(TM_ERR_INVALID_ARG, "info must not be NULL");
  info->K = W->K;
  info->N = W->N;
  info->group = W->group;
  info->dtype = W->dtype;
  info->symmetric = W->symmetric;
  info->device = W->device;
  info->qweight = W->qw;
  info->scales = W->scales;
  info->zeros = W->zeros;
  info->qweight_bytes = W->qw_bytes;
  info->scales_bytes = W->scales_bytes;
  info->zeros_bytes = W->zeros_bytes;
  info->bits = W->bits;
  info->fp8 = W->fp8;
  return TM_OK;
}

tm_status tm_dequant_w4(const tm_packed *W, void *W_out, void *stream) {
  tm_status s = check_handle(W);
  if (s != TM_OK) return s;
  if (W_out == nullptr || !aligned16(W_out))
    return fail(TM_ERR_INVALID_ARG, "W_out must be a 16-byte aligned device pointer");
  if (W->bits == 8) {
    cudaError_t e8 = launch_dequant8(W->qw, W->scales, W->symmetric ? nullptr : W->zeros, W->fp8 != 0,
                                     static_cast<uint16_t *>(W_out), W->K, W->N, W->group, W->dtype == TM_BF16,
                                     static_cast<cudaStream_t>(stream));
    return e8 == cudaSuccess ? TM_OK : fail_cuda(e8, "tm_dequant_w4");
  }
  cudaError_t e = launch_dequant(W->qw, W->scales, W->symmetric ? nullptr : W->zeros,
                                 static_cast<uint16_t *>(W_out), W->K, W->N, W->group,
                                 W->dtype == TM_BF16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "tm_dequant_w4");
  return TM_OK;
}

tm_status tm_select(const tm_packed *W, int M, tm_config *out) {
  tm_status s = check_handle(W);
  if (s != TM_OK) return s;
  if (out == nullptr) return fail(TM_ERR_INVALID_ARG, "out must not be NULL");
  if (M <= 0) return fail(TM_ERR_INVALID_ARG, "M must be positive");
  *out = select_config(W, M, W->device);
  return TM_OK;
}

tm_status tm_gemm_w4a16(const void *A, const tm_packed *W, void *C, int M, int N, int K,
                        void *stream) {
  tm_status s = check_gemm_args(A, W, C, M, N, K);
  if (s != TM_OK || M == 0) return s;
  const tm_config cfg = select_config(W, M, W->device);
  return run_gemm(A, W, C, M, cfg, static_cast<cudaStream_t>(stream));
}

tm_status tm_gemm_w4a16_ex(const void *A, const tm_packed *W, void *C, int M, int N, int K,
                           const tm_config *cfg, void *stream) {
  if (cfg == nullptr) return tm_gemm_w4a16(A, W, C, M, N, K, stream);
  tm_status s = check_gemm_args(A, W, C, M, N, K);
  if (s != TM_OK || M == 0) return s;
  tm_config c = *cfg;
  if (c.kernel == TM_KERNEL_AUTO) c = select_config(W, M, W->device);
  std::string why;
  if (!normalize_config(W, M, &c, &why))
    return fail(TM_ERR_UNSUPPORTED, "variant cannot run this shape: %s", why.c_str());
  return run_gemm(A, W, C, M, c, static_cast<cudaStream_t>(stream));
}

tm_status tm_tc_pipeline(int block_m, int dq_warps, int *stages, int *kblocks_per_stage,
                         int *tmem_slots, int *legal) {
  if (stages == nullptr || kblocks_per_stage == nullptr || tmem_slots == nullptr || legal == nullptr)
    return fail(TM_ERR_INVALID_ARG, "output pointers must not be NULL");
  if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128 && block_m != 256)
    return fail(TM_ERR_INVALID_ARG, "block_m must be 16, 32, 64, 128 or 256");
  tc_pipeline(block_m, stages, kblocks_per_stage, tmem_slots);
  *legal = tc_variant_ok(block_m, dq_warps) ? 1 : 0;
  return TM_OK;
}

tm_status tm_poll_error(void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TM_CUDA(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  int dev = -1;
  tm_status s = current_device(&dev);
  if (s != TM_OK) return s;
  unsigned int *err = nullptr;
  s = error_word(dev, &err);
  if (s != TM_OK) return s;
  unsigned int w[TM_ERR_WORDS] = {};
  TM_CUDA(cudaMemcpy(w, err, sizeof(w), cudaMemcpyDeviceToHost), "cudaMemcpy(error word)");
  // the allocation-free GEMM reports into its own static word: read and
  // clear it too (the first report found is the one described)
  unsigned int ws[TM_ERR_WORDS] = {};
  s = take_static_error(dev, ws);
  if (s != TM_OK) return s;
  if (w[0] == 0 && ws[0] != 0) std::memcpy(w, ws, sizeof(w));
  const unsigned int v = w[0] | ws[0];
  if (v != 0) {
    TM_CUDA(cudaMemset(err, 0, sizeof(w)), "cudaMemset(error word)");
    // a kernel that gave up may have left split-K arrival counters raised
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto &kv : g_ws)
      if (kv.first.first == dev && kv.second.counters)
        TM_CUDA(cudaMemset(kv.second.counters, 0, kv.second.n_counters * sizeof(unsigned int)),
                "cudaMemset(counters)");
  }
  if (v & TM_DEVERR_TIMEOUT)
    return fail(TM_ERR_TIMEOUT,
                "a bounded device wait gave up (site %u, block %u, thread %u, step %u, parity %u)",
                w[2], w[3], w[4], w[5], w[6]);
  if (v & TM_DEVERR_BAD_CODE) return fail(TM_ERR_INVALID_ARG, "a packed code or zero exceeded 15");
  return TM_OK;
}

tm_status tm_selftest_wait_timeout(long long limit_ns, void *stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000LL)
    return fail(TM_ERR_INVALID_ARG, "limit_ns must be in [1000, 1e9]");
  int dev = -1;
  tm_status s = current_device(&dev);
  if (s != TM_OK) return s;
  unsigned int *err = nullptr;
  s = error_word(dev, &err);
  if (s != TM_OK) return s;
  cudaError_t e = launch_wait_selftest(err, static_cast<unsigned long long>(limit_ns),
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "tm_selftest_wait_timeout");
  return TM_OK;
}

// ------------------------------------------------------ decode attention
// 64-token tiles per unit of work (units are handed out dynamically, and
// every unit of a split sequence costs a merge through global memory).
// Measured on GB300 over batch 1..256 at the 8B-class layout: whole
// sequences once there are at least 4 (sequence, KV head) pairs per
// resident CTA; otherwise chunks of 16 tiles, or smaller (down to 4) when
// that would leave resident CTAs idle.  Planned for every sequence at L_max.
static int attn_chunk_tiles(int B, int Hkv, int tiles, int cap) {
  const long long pairs = static_cast<long long>(B) * Hkv;
  if (pairs >= 4LL * cap) return tiles;
  int ct = 16;
  while (ct > 4 && pairs * ((tiles + ct - 1) / ct) < cap) ct /= 2;
  return std::min(ct, tiles);
}

static tm_status encode_kv_map(const uint8_t *cache, long long rows, int row_bytes, CUtensorMap *map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  tm_status s = get_encoder(&enc);
  if (s != TM_OK) return s;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes), 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(cache), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TM_ERR_CUDA, "cuTensorMapEncodeTiled (KV cache) failed (%d)", (int)r);
  return TM_OK;
}

tm_status tm_attn_decode(const void *q, const uint8_t *k_cache, const void *k_scale, const uint8_t *k_zero,
                         const uint8_t *v_cache, const void *v_scale, const uint8_t *v_zero, const int32_t *lens,
                         void *o, int B, int Hq, int Hkv, int head_dim, int L_max, int kv_bits, tm_dtype dtype,
                         float sm_scale, int chunk_tiles, void *stream) {
  if (B < 0 || Hq < 1 || Hkv < 1) return fail(TM_ERR_INVALID_ARG, "B >= 0, Hq >= 1 and Hkv >= 1 required");
  if (Hq % Hkv != 0) return fail(TM_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (Hq / Hkv > 16) return fail(TM_ERR_UNSUPPORTED, "at most 16 query heads per KV head");
  if (B > kAttnMaxBatch) return fail(TM_ERR_UNSUPPORTED, "at most %d sequences per call", kAttnMaxBatch);
  if (head_dim != 128) return fail(TM_ERR_UNSUPPORTED, "head_dim must be 128");
  if (kv_bits != 4 && kv_bits != 8) return fail(TM_ERR_INVALID_ARG, "kv_bits must be 4 or 8");
  if (dtype != TM_F16 && dtype != TM_BF16) return fail(TM_ERR_INVALID_ARG, "dtype must be TM_F16 or TM_BF16");
  if (L_max < 64 || L_max % 64 != 0) return fail(TM_ERR_INVALID_ARG, "L_max must be a positive multiple of 64");
  if (chunk_tiles < 0) return fail(TM_ERR_INVALID_ARG, "chunk_tiles must be >= 0 (0 = automatic)");
  if (!std::isfinite(sm_scale)) return fail(TM_ERR_INVALID_ARG, "sm_scale must be finite");
  const long long rows = static_cast<long long>(B) * Hkv * L_max;
  if (rows > 0x7FFFFFFFLL) return fail(TM_ERR_UNSUPPORTED, "B * Hkv * L_max must be below 2^31");
  if (B == 0) return TM_OK;
  const void *ptrs[] = {q, k_cache, k_scale, k_zero, v_cache, v_scale, v_zero, o};
  for (const void *ptr : ptrs)
    if (ptr == nullptr || !aligned16(ptr))
      return fail(TM_ERR_INVALID_ARG, "q, caches, scales, zeros and o must be non-NULL and 16-byte aligned");
  if (lens == nullptr) return fail(TM_ERR_INVALID_ARG, "lens must not be NULL");
  int dev = -1;
  tm_status s = current_device(&dev);
  if (s != TM_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == TM_BF16;
  const int gq = Hq / Hkv;
  const int occ = attn_decode_ctas_per_sm(bf16, kv_bits, gq, B);
  if (occ < 1) return fail(TM_ERR_CUDA, "decode attention kernel cannot be resident");
  const int cap = sm_count(dev) * occ;
  const int tiles = L_max / 64;
  const int ct = chunk_tiles > 0 ? std::min(chunk_tiles, tiles) : attn_chunk_tiles(B, Hkv, tiles, cap);
  const int n_ch = (tiles + ct - 1) / ct;
  unsigned int *err = nullptr;
  s = error_word(dev, &err);
  if (s != TM_OK) return s;
  AttnArgs a{};
  a.q = static_cast<const uint16_t *>(q);
  a.k_scale = static_cast<const uint16_t *>(k_scale);
  a.v_scale = static_cast<const uint16_t *>(v_scale);
  a.k_zero = k_zero;
  a.v_zero = v_zero;
  a.lens = lens;
  a.o = static_cast<uint16_t *>(o);
  a.err = err;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.L_max = L_max;
  a.chunk_tiles = ct;
  a.n_chunks_max = n_ch;
  a.sm_scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
  a.limit_ns = wait_limit_ns();
  a.pdl = pdl_enabled() ? 1 : 0;
  {
    // partial slots when sequences are split; one arrival counter per
    // (sequence, KV head) plus the two work-ticket counters
    Workspace *ws = nullptr;
    const size_t floats = n_ch > 1 ? static_cast<size_t>(B) * Hkv * n_ch * gq * (128 + 4) : 0;
    s = get_workspace(dev, st, sizeof(float) * floats, static_cast<size_t>(B) * Hkv + 2, &ws);
    if (s != TM_OK) return s;
    a.ws = ws->ws;
    a.counters = ws->counters;
  }
  CUtensorMap kmap, vmap;
  const int row_bytes = 128 * kv_bits / 8;
  s = encode_kv_map(k_cache, rows, row_bytes, &kmap);
  if (s != TM_OK) return s;
  s = encode_kv_map(v_cache, rows, row_bytes, &vmap);
  if (s != TM_OK) return s;
  const long long U = static_cast<long long>(B) * Hkv * n_ch;
  const int grid = static_cast<int>(std::min<long long>(U, cap));
  cudaError_t e = launch_attn_decode(kmap, vmap, a, bf16, kv_bits, grid, st);
  if (e != cudaSuccess) return fail_cuda(e, "tm_attn_decode launch");
  return TM_OK;
}

tm_status tm_attn_decode_plan(int B, int Hq, int Hkv, int L_max, int kv_bits, tm_dtype dtype, int *chunk_tiles,
                              int *grid) {
  if (B < 1 || B > kAttnMaxBatch || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq / Hkv > 16 || L_max < 64 ||
      L_max % 64 != 0 ||
      (kv_bits != 4 && kv_bits != 8))
    return fail(TM_ERR_INVALID_ARG, "invalid decode attention shape");
  int dev = -1;
  tm_status s = current_device(&dev);
  if (s != TM_OK) return s;
  const int occ = attn_decode_ctas_per_sm(dtype == TM_BF16, kv_bits, Hq / Hkv, B);
  if (occ < 1) return fail(TM_ERR_CUDA, "decode attention kernel cannot be resident");
  const int cap = sm_count(dev) * occ;
  const int tiles = L_max / 64;
  const int ct = attn_chunk_tiles(B, Hkv, tiles, cap);
  const long long U = static_cast<long long>(B) * Hkv * ((tiles + ct - 1) / ct);
  if (chunk_tiles) *chunk_tiles = ct;
  if (grid) *grid = static_cast<int>(std::min<long long>(U, cap));
  return TM_OK;
}

// ------------------------------------------------------------- tuning
static bool parse_int(const char *line, const char *key, int *out) {
  const char *p = strstr(line, key);
  if (!p) return false;
  p += strlen(key);
  while (*p == '"' || *p == ':' || *p == ' ') ++p;
  *out = static_cast<int>(strtol(p, nullptr, 10));
  return true;
}

tm_status tm_tune_load(const char *path) {
  if (path == nullptr) return fail(TM_ERR_INVALID_ARG, "path must not be NULL");
  FILE *f = fopen(path, "r");
  if (!f) return fail(TM_ERR_INVALID_ARG, "cannot open %s", path);
  char line[512];
  std::lock_guard<std::mutex> lk(g_mu);
  while (fgets(line, sizeof(line), f)) {
    TuneKey k{};
    TuneVal v{};
    int M = 0;
    if (parse_int(line, "\"N\"", &k.N) && parse_int(line, "\"K\"", &k.K) &&
        parse_int(line, "\"group\"", &k.group) && parse_int(line, "\"dtype\"", &k.dtype) &&
        parse_int(line, "\"sym\"", &k.sym) && parse_int(line, "\"M\"", &M) && M > 0 &&
        parse_int(line, "\"kernel\"", &v.cfg.kernel) &&
        parse_int(line, "\"block_m\"", &v.cfg.block_m) &&
        parse_int(line, "\"split_k\"", &v.cfg.split_k) &&
        parse_int(line, "\"dq_warps\"", &v.cfg.dq_warps)) {
      k.mb = m_bucket(M);
      if (!parse_int(line, "\"fmt\"", &k.fmt)) k.fmt = 0;   // tables without it: int4
      v.M = M;
      g_tune[k] = v;
    }
  }
  fclose(f);
  return TM_OK;
}

tm_status tm_tune_save(const char *path) {
  if (path == nullptr) return fail(TM_ERR_INVALID_ARG, "path must not be NULL");
  FILE *f = fopen(path, "w");
  if (!f) return fail(TM_ERR_INVALID_ARG, "cannot write %s", path);
  std::lock_guard<std::mutex> lk(g_mu);
  for (const auto &kv : g_tune) {
    const TuneKey &k = kv.first;
    const TuneVal &v = kv.second;
    fprintf(f,
            "{\"N\": %d, \"K\": %d, \"group\": %d, \"dtype\": %d, \"sym\": %d, \"fmt\": %d, \"M\": %d, "
            "\"m_bucket\": %d, \"kernel\": %d, \"block_m\": %d, \"split_k\": %d, \"dq_warps\": %d, "
            "\"us\": %.3f}\n",
            k.N, k.K, k.group, k.dtype, k.sym, k.fmt, v.M, k.mb, v.cfg.kernel, v.cfg.block_m, v.cfg.split_k,
            v.cfg.dq_warps, v.us);
  }
  fclose(f);
  return TM_OK;
}

}  // extern "C"

static void load_tune_env_once() {
  static std::once_flag once;
  std::call_once(once, [] {
    const char *p = getenv("TM_TUNE_CACHE");
    if (p && *p) {
      FILE *f = fopen(p, "r");
      if (f) {
        fclose(f);
        tm_tune_load(p);
      }
    }
  });
}

// Legal variants worth measuring for this shape, the built-in choice first.
static std::vector<tm_config> candidates(const tm_packed *W, int M, int dev) {
  std::vector<tm_config> out;
  const int KB = W->K / 64;
  const int sms = sm_count(dev);
  auto add = [&](tm_config c) {
    if (!normalize_config(W, M, &c, nullptr)) return;
    for (const tm_config &o : out)
      if (o.kernel == c.kernel && o.block_m == c.block_m && o.split_k == c.split_k &&
          o.dq_warps == c.dq_warps)
        return;
    out.push_back(c);
  };
  add(default_config(W, M, dev));
  const int splits[] = {1, 2, 3, 4, 6, 8, 12, 16, 24, 32};
  if (M <= 16) {
    for (int s = 1; s <= 8; ++s) add(tm_config{TM_KERNEL_DECODE_MMA, 0, s, 4});
    for (int s = 1; s <= 2; ++s) add(tm_config{TM_KERNEL_DECODE_MMA, 0, s, 8});
    add(tm_config{TM_KERNEL_DECODE_MMA, 0, 1, 16});
    for (int s : {2, 4, 6, 8, 12, 16}) add(tm_config{TM_KERNEL_DECODE_MMA, 0, s, 1});
    for (int s : {2, 4, 8}) add(tm_config{TM_KERNEL_DECODE_MMA, 0, s, 2});
  }
  if (M <= 8) {
    for (int s : splits) add(tm_config{TM_KERNEL_GEMV, 0, s, 0});
  }
  if (M <= 16) {
    for (int s : splits) add(tm_config{TM_KERNEL_GEMV, 0, s, 1});
  }
  for (int bm : {16, 32, 64}) {
    if (bm > 16 && bm / 2 >= M) continue;
    for (int dq : {4, 8, 12, 16}) add(tm_config{TM_KERNEL_TC_DECODE, bm, 1, dq});
  }
  for (int bm : {16, 32, 64, 128, 256}) {
    if (bm > 16 && bm / 2 >= M) continue;        // at most one mostly empty tile size
    const int tiles = (W->N / 128) * ((M + bm - 1) / bm);
    for (int s : splits) {
      if (s > KB || (s > 1 && tiles * s > 8 * sms)) continue;
      for (int dq : {4, 8, 16}) add(tm_config{TM_KERNEL_TC, bm, s, dq});
    }
  }
  return out;
}

// A packed weight's device storage copied into fresh buffers (the tuner's
// rotated copies, so that back-to-back launches read their weights from HBM).
static tm_status clone_packed(const tm_packed *W, cudaStream_t st, tm_packed *out) {
  *out = *W;
  out->qw = nullptr;
  out->scales = nullptr;
  out->zeros = nullptr;
  TM_CUDA(cudaMalloc(reinterpret_cast<void **>(&out->qw), W->qw_bytes), "cudaMalloc(tune copy)");
  TM_CUDA(cudaMalloc(reinterpret_cast<void **>(&out->scales), W->scales_bytes), "cudaMalloc(tune copy)");
  if (W->zeros)
    TM_CUDA(cudaMalloc(reinterpret_cast<void **>(&out->zeros), W->zeros_bytes), "cudaMalloc(tune copy)");
  TM_CUDA(cudaMemcpyAsync(out->qw, W->qw, W->qw_bytes, cudaMemcpyDeviceToDevice, st), "copy");
  TM_CUDA(cudaMemcpyAsync(out->scales, W->scales, W->scales_bytes, cudaMemcpyDeviceToDevice, st), "copy");
  if (W->zeros)
    TM_CUDA(cudaMemcpyAsync(out->zeros, W->zeros, W->zeros_bytes, cudaMemcpyDeviceToDevice, st), "copy");
  return TM_OK;
}

// Seconds per launch of variant c: `launches` launches over the rotated
// weights, captured in one CUDA graph (back to back, with programmatic
// dependent launch as in the caller's graphs), median of three replays.
// Returns a negative value if the variant did not run.
static double time_variant_graph(const void *A, const std::vector<const tm_packed *> &Ws, void *C,
                                 int M, const tm_config &c, int launches, cudaStream_t st,
                                 cudaEvent_t e0, cudaEvent_t e1) {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return -1.0;
  bool ok = true;
  for (int i = 0; i < launches && ok; ++i)
    ok = run_gemm(A, Ws[i % Ws.size()], C, M, c, st) == TM_OK;
  if (cudaStreamEndCapture(st, &graph) != cudaSuccess || !ok) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return -1.0;
  }
  if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
    cudaGraphDestroy(graph);
    cudaGetLastError();
    return -1.0;
  }
  float ms[3] = {};
  bool good = cudaGraphLaunch(exec, st) == cudaSuccess;   // warm replay
  for (int r = 0; r < 3 && good; ++r) {
    good = cudaEventRecord(e0, st) == cudaSuccess && cudaGraphLaunch(exec, st) == cudaSuccess &&
           cudaEventRecord(e1, st) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
           cudaEventElapsedTime(&ms[r], e0, e1) == cudaSuccess;
  }
  cudaGraphExecDestroy(exec);
  cudaGraphDestroy(graph);
  if (!good) {
    cudaGetLastError();
    return -1.0;
  }
  std::sort(ms, ms + 3);
  return ms[1] * 1e-3 / launches;
}

// The tuner's own stream on device `dev` (non-blocking, created once): the
// caller's stream may be the legacy default stream, which cannot be
// captured into a graph.
static tm_status tune_stream(int dev, cudaStream_t *out) {
  static cudaStream_t streams[kMaxDevices] = {};
  std::lock_guard<std::mutex> lk(g_mu);
  if (streams[dev] == nullptr)
    TM_CUDA(cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking), "cudaStreamCreate(tuner)");
  *out = streams[dev];
  return TM_OK;
}

extern "C" tm_status tm_tune(const int *Ms, int nM, const tm_packed *W, void *stream,
                             tm_config *best_out) {
  tm_status s = check_handle(W);
  if (s != TM_OK) return s;
  if (Ms == nullptr || nM <= 0) return fail(TM_ERR_INVALID_ARG, "Ms must hold nM > 0 values");
  cudaStream_t user_st = static_cast<cudaStream_t>(stream);
  if (stream_capturing(user_st)) return fail(TM_ERR_UNSUPPORTED, "tm_tune cannot run during capture");
  // everything below runs on the tuner's stream, after the caller's work
  TM_CUDA(cudaStreamSynchronize(user_st), "cudaStreamSynchronize");
  cudaStream_t st = nullptr;
  s = tune_stream(W->device, &st);
  if (s != TM_OK) return s;
  int maxM = 0;
  for (int i = 0; i < nM; ++i) {
    if (Ms[i] <= 0) return fail(TM_ERR_INVALID_ARG, "Ms values must be positive");
    maxM = std::max(maxM, Ms[i]);
  }
  int l2 = 0;
  cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, W->device);
  const size_t wbytes = W->qw_bytes + W->scales_bytes + W->zeros_bytes;
  // enough distinct copies that a launch never finds its weights in L2
  const int ncopies = static_cast<int>(std::min<size_t>(8, (2 * static_cast<size_t>(l2)) / wbytes + 2));
  void *A = nullptr, *C = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  std::vector<tm_packed> copies(ncopies - 1);
  std::vector<const tm_packed *> Ws{W};
  auto cleanup = [&]() {
    cudaStreamSynchronize(st);
    if (A) cudaFree(A);
    if (C) cudaFree(C);
    for (tm_packed &c : copies) {
      if (c.qw) cudaFree(c.qw);
      if (c.scales) cudaFree(c.scales);
      if (c.zeros) cudaFree(c.zeros);
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
  };
  cudaError_t e = cudaMalloc(&A, static_cast<size_t>(maxM) * W->K * 2);
  if (e == cudaSuccess) e = cudaMalloc(&C, static_cast<size_t>(maxM) * W->N * 2);
  if (e == cudaSuccess) e = cudaMemsetAsync(A, 0, static_cast<size_t>(maxM) * W->K * 2, st);
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e != cudaSuccess) {
    cleanup();
    return fail_cuda(e, "tm_tune setup");
  }
  for (tm_packed &c : copies) {
    s = clone_packed(W, st, &c);
    if (s != TM_OK) {
      cleanup();
      return s;
    }
    Ws.push_back(&c);
  }
  for (int i = 0; i < nM; ++i) {
    const int M = Ms[i];
    std::vector<tm_config> cands = candidates(W, M, W->device);
    double best_s = 1e30;
    tm_config best{};
    for (const tm_config &c : cands) {
      // eager warm-up on every copy (sizes the split-K workspace outside
      // capture) and a first estimate of the launch time
      bool ran = true;
      for (size_t j = 0; j < Ws.size() && ran; ++j) ran = run_gemm(A, Ws[j], C, M, c, st) == TM_OK;
      if (!ran) continue;
      float ms = 0.f;
      if (cudaEventRecord(e0, st) != cudaSuccess || run_gemm(A, Ws[0], C, M, c, st) != TM_OK ||
          cudaEventRecord(e1, st) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
          cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
        continue;
      // about 0.3 ms of work per graph, 4..24 launches
      const int launches = std::max(4, std::min(24, static_cast<int>(0.3 / std::max(ms, 1e-3f))));
      const double t = time_variant_graph(A, Ws, C, M, c, launches, st, e0, e1);
      if (t <= 0) continue;
      // earlier candidates (the built-in choice first) keep their place
      // unless a later one is at least 2% faster: stable picks under noise
      if (t < best_s * 0.98) {
        best_s = t;
        best = c;
      }
    }
    if (best_s >= 1e29) {
      cleanup();
      return fail(TM_ERR_CUDA, "no variant ran for M=%d", M);
    }
    {
      std::lock_guard<std::mutex> lk(g_mu);
      g_tune[tune_key(W, M)] = TuneVal{best, best_s * 1e6, M};
    }
    if (best_out) best_out[i] = best;
  }
  cleanup();
  tm_status perr = tm_poll_error(st);
  if (perr != TM_OK) return perr;
  const char *p = getenv("TM_TUNE_CACHE");
  if (p && *p) return tm_tune_save(p);
  return TM_OK;
}

// ======================================================================
// GEMM without any device allocation.
//
// For callers that cannot allocate device memory: an allocator-less
// embedding (the host application owns every byte of the GPU through its
// own pool and forbids cudaMalloc behind its back).  The split-K partials,
// the tile arrival counters and the device error words live in file-scope
// static __device__ arrays of fixed size, loaded with the library and held
// by every GPU that loads it until the process exits.  In host code the
// array names are host-side stand-ins, not device addresses, so their device
// addresses are fetched once per device with cudaGetSymbolAddress.
// ======================================================================

static constexpr size_t kStaticWsFloats = static_cast<size_t>(2) << 20;  // 8 MiB of partials
static constexpr size_t kStaticCounters = 16384;                          // 64 KiB of counters

static __device__ __align__(256) float g_static_ws[kStaticWsFloats];
static __device__ __align__(256) unsigned int g_static_counters[kStaticCounters];
static __device__ __align__(256) unsigned int g_static_err[TM_ERR_WORDS];

struct StaticScratch {
  bool ready = false;
  float *ws = nullptr;
  unsigned int *counters = nullptr;
  unsigned int *err = nullptr;
};
static StaticScratch g_static[kMaxDevices];

// Device addresses of the static arrays on device `dev` (which must be
// current); fetched on the first call on that device.
static tm_status static_scratch(int dev, StaticScratch **out) {
  std::lock_guard<std::mutex> lk(g_mu);
  StaticScratch &s = g_static[dev];
  if (!s.ready) {
    void *p = nullptr;
    TM_CUDA(cudaGetSymbolAddress(&p, g_static_ws), "cudaGetSymbolAddress(split-K scratch)");
    s.ws = static_cast<float *>(p);
    TM_CUDA(cudaGetSymbolAddress(&p, g_static_counters), "cudaGetSymbolAddress(counters)");
    s.counters = static_cast<unsigned int *>(p);
    TM_CUDA(cudaGetSymbolAddress(&p, g_static_err), "cudaGetSymbolAddress(error words)");
    s.err = static_cast<unsigned int *>(p);
    s.ready = true;
  }
  *out = &s;
  return TM_OK;
}

static tm_status take_static_error(int dev, unsigned int (&w)[TM_ERR_WORDS]) {
  unsigned int *err = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_static[dev].ready) err = g_static[dev].err;
  }
  std::memset(w, 0, sizeof(w));
  if (err == nullptr) return TM_OK;
  TM_CUDA(cudaMemcpy(w, err, sizeof(w), cudaMemcpyDeviceToHost), "cudaMemcpy(static error word)");
  if (w[0] != 0) TM_CUDA(cudaMemset(err, 0, sizeof(w)), "cudaMemset(static error word)");
  return TM_OK;
}

extern "C" tm_status tm_gemm_w4a16_noalloc(const void *A, const tm_packed *W, void *C, int M, int N,
                                           int K, void *stream) {
  tm_status s = check_gemm_args(A, W, C, M, N, K);
  if (s != TM_OK || M == 0) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  StaticScratch *sc = nullptr;
  s = static_scratch(W->device, &sc);
  if (s != TM_OK) return s;
  const tm_config cfg = select_config(W, M, W->device);
  GemmArgs a{};
  a.qw = W->qw;
  a.scales = W->scales;
  a.zeros = W->symmetric ? nullptr : W->zeros;
  a.A = static_cast<const uint16_t *>(A);
  a.C = static_cast<uint16_t *>(C);
  a.err = sc->err;
  a.M = M;
  a.N = W->N;
  a.K = W->K;
  a.group = W->group;
  a.wbits = W->bits;
  a.fp8 = W->fp8;
  int dec_grid = 0;
  size_t ws_floats = 0, tiles = 0;
  plan_work(W, M, cfg, &a, &dec_grid, &ws_floats, &tiles);
  a.limit_ns = wait_limit_ns();
  a.pdl = pdl_enabled() ? 1 : 0;
  if (ws_floats > 0) {
    if (ws_floats > kStaticWsFloats || tiles > kStaticCounters)
      return fail(TM_ERR_UNSUPPORTED,
                  "tm_gemm_w4a16_noalloc: this shape needs %zu bytes of split-K scratch and %zu "
                  "counters; the static scratch holds %zu bytes and %zu counters",
                  ws_floats * sizeof(float), tiles, kStaticWsFloats * sizeof(float),
                  kStaticCounters);
    // the counters must start at zero (a kernel that gave up may have left
    // some raised); clearing is stream-ordered and allocates nothing
    TM_CUDA(cudaMemsetAsync(sc->counters, 0, tiles * sizeof(unsigned int), st),
            "cudaMemsetAsync(counters)");
    a.ws = sc->ws;
    a.counters = sc->counters;
  }
  return launch_planned(A, W, M, cfg, a, dec_grid, st, "tm_gemm_w4a16_noalloc launch");
}

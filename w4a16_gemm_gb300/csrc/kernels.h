// kernels.h -- launch entry points of the device kernels (host-callable).
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tmw4 {

// Source layouts of the repack and zero packing (see pack.cu).
enum SrcLayout { SRC_U8 = 0, SRC_AWQ = 1, SRC_GPTQ = 2 };
cudaError_t launch_repack(const void *q, uint8_t *qw, int K, int N, int src, unsigned int *err,
                          cudaStream_t st);
// rows packed group rows, each from source row / rep; offset added to zeros
cudaError_t launch_pack_zeros(const void *z, uint8_t *zp, int rows, int N, int rep, int src, int offset,
                              unsigned int *err, cudaStream_t st);
cudaError_t launch_pack_scales(const uint16_t *s, uint16_t *sp, int rows, int N, int rep, cudaStream_t st);
cudaError_t launch_dequant(const uint8_t *qw, const uint16_t *scales, const uint8_t *zeros,
                           uint16_t *out, int K, int N, int group, bool bf16, cudaStream_t st);
// 8-bit weights (int8 codes with byte zeros, or FP8 E4M3 codes): repack of
// u8 [K][N] codes, byte zeros, dequant-only (see pack.cu for the layout).
cudaError_t launch_repack8(const uint8_t *q, uint8_t *qw, int K, int N, cudaStream_t st);
cudaError_t launch_pack_zeros8(const uint8_t *z, uint8_t *zp, int rows, int N, int rep, cudaStream_t st);
cudaError_t launch_dequant8(const uint8_t *qw, const uint16_t *scales, const uint8_t *zeros, bool fp8,
                            uint16_t *out, int K, int N, int group, bool bf16, cudaStream_t st);

// Shared arguments of the GEMM kernels.  ws/counters are the split-K
// workspace (partials [splits][M][N] fp32 and one self-resetting arrival
// counter per output tile); unused when splits == 1.
struct GemmArgs {
  const uint8_t *qw;
  const uint16_t *scales;
  const uint8_t *zeros;  // nullptr: symmetric
  const uint16_t *A;
  uint16_t *C;
  float *ws;
  unsigned int *counters;
  unsigned int *err;
  int M, N, K, group;
  int wbits;         // bits per weight code: 4, or 8 (int8 with byte zeros, or FP8)
  int fp8;           // 8-bit codes are FP8 E4M3 (no zeros)
  int splits;
  int kb_per_split;  // 64-wide K blocks per split (a multiple of the TC stage's k-blocks)
  int act_map_3d;    // TC: the activation tensor map is 3-D (64 x M x K/64)
  int ws_slots;      // TC_DECODE: fp32 partial slots per tile in ws (stream-K contributors)
  unsigned long long limit_ns;
  // Host side only: launch with programmatic stream serialization, so the
  // kernel's prologue and weight loads overlap the previous kernel's tail.
  // Every GEMM kernel calls pdl_wait() before it reads A or touches C, the
  // split-K workspace or its counters.
  int pdl;
  // Debug builds compiled with -DTMW4_TRACE record per-stage SM cycle
  // stamps of CTA (0,0,0) here ([8][256] slots); nullptr otherwise.
  long long *trace;
};

// Decode attention over a low-bit KV cache (attn_decode.cu).  q, o
// [B][Hq][128]; cache rows [B][Hkv][L_max][128 * bits / 8] (K and V, through
// the tensor maps); scales [B][Hkv][L_max] 16-bit; zeros [B][Hkv][L_max]
// bytes; lens [B] (device).  ws holds one 132-float slot (O[128], m, l) per
// (sequence, KV head, chunk, query head of the group); counters one
// self-resetting arrival count per (sequence, KV head).
struct AttnArgs {
  const uint16_t *q;
  const uint16_t *k_scale;
  const uint16_t *v_scale;
  const uint8_t *k_zero;
  const uint8_t *v_zero;
  const int *lens;
  uint16_t *o;
  float *ws;
  unsigned int *counters;
  unsigned int *err;
  int B, Hq, Hkv, L_max;
  int chunk_tiles;    // 64-token tiles per unit of work
  int n_chunks_max;   // ceil(L_max / (64 * chunk_tiles))
  float sm_scale_log2;
  unsigned long long limit_ns;
  int pdl;
};
constexpr int kAttnMaxBatch = 4096;   // sequences per call (the unit scan lives in shared memory)
size_t attn_decode_smem_bytes(int bits, int gq, int B);
int attn_decode_ctas_per_sm(bool bf16, int bits, int gq, int B);
cudaError_t launch_attn_decode(const CUtensorMap &kmap, const CUtensorMap &vmap, const AttnArgs &a, bool bf16,
                               int bits, int grid, cudaStream_t st);

// Launch kern<<<grid, block, smem, st>>>(args...), with programmatic stream
// serialization when pdl is set (see GemmArgs::pdl).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  unsigned n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The same with thread-block clusters of cluster_y CTAs along grid.y.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                         cudaStream_t st, bool pdl, unsigned cluster_y, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;
  attr[n].val.clusterDim.x = 1;
  attr[n].val.clusterDim.y = cluster_y;
  attr[n].val.clusterDim.z = 1;
  ++n;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Opts kernel Kern into `bytes` of dynamic shared memory on the current
// device.  The attribute belongs to the device's context, so it is set once
// per device; concurrent first calls from several host threads are safe.
// `bytes` must be the same on every call for a given kernel.
constexpr int kMaxOptinDevices = 64;
template <auto Kern>
inline cudaError_t smem_optin(int bytes) {
  static std::once_flag once[kMaxOptinDevices];
  static cudaError_t result[kMaxOptinDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxOptinDevices) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    result[dev] = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
  return result[dev];
}

// smem_optin, and clusters of up to 16 CTAs (beyond the portable 8).
template <auto Kern>
inline cudaError_t cluster_optin(int bytes) {
  static std::once_flag once[kMaxOptinDevices];
  static cudaError_t result[kMaxOptinDevices];
  int dev = 0;
  cudaError_t e = smem_optin<Kern>(bytes);
  if (e != cudaSuccess) return e;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::call_once(once[dev], [&] {
    result[dev] = cudaFuncSetAttribute(Kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  return result[dev];
}

// GEMV: rows_tmpl in {1,2,4,8} >= M on the CUDA cores (mma = false), or
// 8 / 16 >= M with register-operand tensor-core MMAs (mma = true).  Shared
// memory bytes of each mode:
size_t gemv_smem_bytes(int rows_tmpl, int kb_per_split);
size_t gemv_mma_smem_bytes(int nt8, int kb_per_split, int group);
cudaError_t launch_gemv(const GemmArgs &a, bool bf16, int rows_tmpl, bool mma, cudaStream_t st);

// tcgen05 kernel.  block_m in {16,32,64,128,256}, dq_warps in {4,8}.
size_t tc_smem_bytes(int block_m);
int tc_stages(int block_m);
int tc_kblocks_per_stage(int block_m);
// Pipeline geometry of the tcgen05 kernel for a legal block_m.
void tc_pipeline(int block_m, int *stages, int *kbs, int *tmem_slots);
// Whether (block_m, dq_warps) is a legal tcgen05 variant (see tc_gemm.cu).
bool tc_variant_ok(int block_m, int dq_warps, int wbits = 4);
cudaError_t launch_tc(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int block_m,
                      int dq_warps, cudaStream_t st);

// tcgen05 decode kernel: persistent, stream-K; block_m in {16,32,64},
// dq_warps in {4,8,12} (see tc_decode.cu).  tc_decode_plan gives the grid,
// the tile count (split-K counters) and the partial slots per tile.
bool tc_decode_ok(int block_m, int dq_warps);
int tc_decode_slots(int block_m, int dq_warps);
int tc_decode_kblocks_per_stage();   // 64-K blocks per activation box
void tc_decode_pipeline(int block_m, int dq_warps, int *weight_stages, int *act_stages_per_wg,
                        int *tmem_slots_per_wg);
void tc_decode_plan(int M, int N, int K, int block_m, int sms, int *grid, long long *tiles,
                    int *ws_slots);
cudaError_t launch_tc_decode(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int block_m,
                             int dq_warps, int grid, cudaStream_t st);

// Kernel with register-operand tensor-core MMAs (M <= 16; decode_mma_nt8(M)
// n8 tiles of activation rows, 0 if M is too large; kgroups = 1, 2 or 4
// K-groups of four consumer warps per CTA).  Stream-K mode:
// decode_mma_ctas_per_sm gives the resident CTAs per SM of the instantiation
// for (bf16, M, group, kgroups); decode_mma_plan the grid for at most max_ctas CTAs,
// the tile count (split-K counters) and the fp32 partial slots per tile (1:
// no tile is cut between CTAs).  Cluster mode: decode_mma_cluster_split
// turns a requested cluster size into the group-aligned 64-K blocks per
// split and the cluster size that covers K with them (0 if no cluster of
// that size can be resident).
int decode_mma_nt8(int M);
int decode_mma_ctas_per_sm(bool bf16, int M, int group, int kgroups, int wbits = 4);
void decode_mma_plan(int M, int N, int K, int group, int max_ctas, int *grid, long long *tiles,
                     int *slots);
int decode_mma_cluster_split(bool bf16, int M, int K, int group, int kgroups, int requested, int *kb_per_split,
                             int wbits = 4);
// tmap_a: activation tensor map with box 64 x (8 * decode_mma_nt8(M)) and the
// 128-byte swizzle (3-D with one 64-K block per copy, or 2-D).  cluster = 0:
// stream-K over `grid` CTAs; cluster = S > 0: grid (grid tiles, S) in
// clusters of S with a.kb_per_split blocks per split (kgroups 1 or 2).
cudaError_t launch_decode_mma(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int kgroups, int grid,
                              int cluster, cudaStream_t st);
// The code-width instantiations behind the three calls above (WB = 4 or 8 bits).
template <int WB>
cudaError_t dm_launch_wb(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int kgroups, int grid, int cluster,
                         cudaStream_t st);
template <int WB>
int dm_ctas_per_sm_wb(bool bf16, int M, int group, int kgroups);
template <int WB>
int dm_cluster_split_wb(bool bf16, int M, int K, int group, int kgroups, int requested, int *kb_per_split);

// Bounded-wait self-test kernel.
cudaError_t launch_wait_selftest(unsigned int *err, unsigned long long limit_ns, cudaStream_t st);

}  // namespace tmw4

/*
 * tmw4.h -- C ABI of the GB300 (sm_103a) W4A16 GEMM library (libtmw4.so).
 *
 * The library implements the mixed-precision GEMM pipeline of the TurboMind
 * engine ("Efficient Mixed-Precision Large Language Model Inference with
 * TurboMind", arXiv 2508.15601; abstract: a GEMM pipeline in two parts, an
 * offline packing of the weights and an accelerated online multiply):
 *
 *   offline:  tm_pack_w4     int4 codes + scales + zeros -> packed weight
 *             (tm_pack_awq / tm_pack_gptq: the same from AWQ / GPTQ int32
 *             packed checkpoints)
 *   online:   tm_gemm_w4a16  C[M,N] = A[M,K] * W[K,N],
 *                            W[k,n] = T(s[k/G,n] * (q[k,n] - z[k/G,n]))
 *   (tm_pack_w8 / tm_pack_fp8: 8-bit weights on the same pipeline)
 *
 * Beside it, the decode kernel of the engine's attention pipeline:
 *   tm_attn_decode  one query token per sequence against an 8- or 4-bit KV
 *                   cache dequantized the same way, per token and KV head
 *
 * Conventions used by every call:
 *   - All matrices are row-major.  The logical weight W is [K, N]; A is
 *     [M, K]; C is [M, N]; q is [K, N] (one code 0..15 per byte); scales and
 *     zeros are [K/G, N].  T is the 16-bit float type of A, scales and C.
 *   - "device" pointers are CUDA device addresses on the current device;
 *     "host" pointers are ordinary CPU memory.  Streams are passed as
 *     `void *` holding a cudaStream_t (NULL = the legacy default stream).
 *   - Every call is stream-ordered and asynchronous unless stated; none
 *     synchronises the device.  No call throws, exits or traps.  On a
 *     non-OK status, tm_last_error() returns a message for the calling
 *     thread.
 *   - Conditions found on the device (a code byte above 15, a bounded wait
 *     that gave up) are recorded in a per-device error word and reported by
 *     tm_poll_error().
 *   - GEMM kernels are launched with programmatic stream serialization
 *     (programmatic dependent launch): a GEMM may start while the previous
 *     kernel in the stream is finishing and stream its packed weights at
 *     once, but it reads A and writes C (and its split-K scratch) only after
 *     that kernel has completed and its writes are visible.  Stream order is
 *     therefore kept for A and C; the packed weight must not be modified by
 *     the previous kernel.  Setting the environment variable TM_PDL=0
 *     before the first GEMM launches every kernel plainly.
 */
#ifndef TMW4_H
#define TMW4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TM_OK = 0,
  TM_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or handle        */
  TM_ERR_UNSUPPORTED = 2, /* valid request this build cannot run           */
  TM_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed             */
  TM_ERR_OOM = 4,         /* device allocation failed                       */
  TM_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up            */
} tm_status;

typedef enum { TM_F16 = 0, TM_BF16 = 1 } tm_dtype;

/* Kernel families (tm_config.kernel). */
enum {
  TM_KERNEL_AUTO = 0,     /* pick from the tuned table, else the built-in rule */
  TM_KERNEL_GEMV = 1,     /* split-K GEMV: 64-column strips, eight warps over K;
                              dq_warps 0: CUDA-core FMAs, M <= 8; dq_warps 1:
                              register-operand tensor-core MMAs, M <= 16 */
  TM_KERNEL_TC = 2,       /* tcgen05/TMEM kernel, weights staged by TMA        */
  TM_KERNEL_TC_DECODE = 3, /* tcgen05/TMEM kernel for small M (block_m 16..64):
                              persistent stream-K grid, weights staged in shared
                              memory by bulk copies, dequantized into TMEM */
  TM_KERNEL_DECODE_MMA = 4 /* kernel for M <= 16: weights streamed through
                              shared memory by bulk copies of a producer warp,
                              dequantized in registers and multiplied by
                              register-operand tensor-core MMAs (mma.sync),
                              group scale applied in fp32.  Two work splits,
                              chosen by dq_warps:
                                4, 8, 16 (0 = 4)  persistent stream-K grid
                                   of CTAs with that many consumer warps;
                                   split_k = CTAs per SM (0: all that fit);
                                1, 2  one thread-block cluster of split_k
                                   CTAs (1..16; fewer for large M) per
                                   128-column tile, each with 4 or 8
                                   consumer warps and an equal group-aligned
                                   K range; partial sums added through
                                   distributed shared memory (no
                                   workspace) */
};

/* A kernel variant: family, rows of A per CTA tile (TC: 16, 32, 64, 128 or
 * 256; TC_DECODE: 16, 32 or 64; GEMV: ignored) and the number of K splits
 * (>= 1). */
typedef struct {
  int32_t kernel;
  int32_t block_m;
  int32_t split_k;
  int32_t dq_warps; /* TC: dequant warps per CTA, 4, 8 or 16 (0 = default);
                       each group of 4 dequantizes every (dq_warps/4)-th stage;
                       TC_DECODE: 4, 8 or 12 dequant warps; DECODE_MMA: the
                       work split and consumer warps (see above) */
} tm_config;

/* Opaque packed weight, owned by the library until tm_packed_free. */
typedef struct tm_packed tm_packed;

/* Read-only view of a packed weight (for inspection and tests).
 *
 * Packed weight layout (the library's own Blackwell order; the pages'
 * packing -- pith.science review, Figures 6 and 7 -- permutes each thread's
 * eight int4 values into MMA order and stores fragments in load order):
 *   qweight: K*N/2 bytes.  Columns form 128-wide tiles; tile nt and K-block
 *     kb (64 values of K) is a 4096-byte block at byte (nt*(K/64) + kb)*4096,
 *     so all of a tile's K is contiguous.  The block holds two 2048-byte
 *     atoms, a = 0 for the tile's columns [0,64), a = 1 for [64,128).  An
 *     atom holds 512 little-endian 32-bit words; word h*256 + nl*4 + j
 *     (h in {0,1}, nl in [0,64), j in [0,4)) holds
 *     q[64kb + 8(4h+j) + e][128nt + 64a + nl] for e = 0..7, value e in bits
 *     [4p, 4p+4) with p = (0,4,1,5,2,6,3,7)[e] -- the word order of
 *     pith.science review Figures 23/24 (e7 e5 e3 e1 e6 e4 e2 e0).  Every
 *     16-byte chunk is 32 consecutive K values of one column.
 *   scales: tile-major [N/128][K/G][128] 16-bit values of type `dtype`.
 *   zeros:  tile-major [N/128][K/G][64] bytes, each byte two columns (even
 *     column in the low nibble); NULL for the symmetric format (zero 8). */
typedef struct {
  int32_t K, N, group; /* group: the one the kernels run with (32, 64 or 128;
                          a coarser source group is repeated, see tm_pack_w4) */
  int32_t dtype;     /* tm_dtype */
  int32_t symmetric; /* 1: no stored zeros, zero point 8 */
  int32_t device;
  const void *qweight; /* device */
  const void *scales;  /* device */
  const void *zeros;   /* device, NULL if symmetric */
  size_t qweight_bytes, scales_bytes, zeros_bytes;
  int32_t bits;        /* bits per weight code: 4, or 8 (tm_pack_w8 / tm_pack_fp8) */
  int32_t fp8;         /* 1: the 8-bit codes are FP8 E4M3 */
} tm_packed_info;

/* Offline repack (TurboMind paper, arXiv abstract: "offline weight
 * packing"; pith.science review, Figures 6/7: steps (i)-(iv) load, place,
 * permute and store fragments).
 *   q      device, [K][N] uint8 codes 0..15 (a code > 15 is masked to 4
 *          bits and reported by tm_poll_error as TM_ERR_INVALID_ARG)
 *   scales device, [K/group][N] 16-bit values of type dtype
 *   zeros  device, [K/group][N] uint8 zero points 0..15, or NULL for the
 *          symmetric format (zero point 8)
 *   K % group == 0, K % 64 == 0, group 32 or a positive multiple of 64
 *   (per-channel weights: group = K), N % 128 == 0, K, N > 0; all pointers
 *   16-byte aligned.  Groups of 32, 64 and 128 are kept; a coarser group is
 *   stored as groups of 128 (of 64 if it is an odd multiple of 64) with its
 *   scale and zero repeated, which leaves every dequantized weight
 *   unchanged.  Groups of 32 run on the TC kernel and the CUDA-core GEMV
 *   only (the other kernels report TM_ERR_UNSUPPORTED for them).
 *   On TM_OK *out receives a new handle; the inputs may be reused once
 *   `stream` has passed this call.  The handle's storage is allocated with
 *   cudaMallocAsync on `stream`. */
tm_status tm_pack_w4(const uint8_t *q, const void *scales, const uint8_t *zeros, int K, int N,
                     int group, tm_dtype dtype, void *stream, tm_packed **out);

/* The same repack, reading the int4 codes and zero points straight from the
 * int32-packed layouts in which AWQ and GPTQ checkpoints are distributed
 * (the pages' evaluated models are AWQ checkpoints: pith.science review,
 * Figure 11, "Qwen3 8B AWQ"), without an intermediate [K][N] byte array.
 * Dequantization is the same, W = T(s * (q - z)).
 *
 * AWQ ("GEMM" layout):
 *   qweight device, int32 [K][N/8]: word (k, j) holds columns 8j + c of row
 *           k, column offset c in nibble p(c) with p = (0,4,1,5,2,6,3,7)
 *           (even columns in the low four nibbles, odd ones in the high four)
 *   qzeros  device, int32 [K/group][N/8], the same packing, or NULL
 *           (symmetric, zero point 8)
 *   scales  device, [K/group][N] of type dtype
 * GPTQ:
 *   qweight device, int32 [K/8][N]: word (r, n) holds rows 8r + i of column
 *           n in nibble i
 *   qzeros  device, int32 [K/group][N/8]: column 8c + i in nibble i of word
 *           (g, c), or NULL (symmetric); zero_offset (0 or 1) is added to
 *           every stored zero (files of the original GPTQ format store
 *           zero - 1); a resulting zero above 15 is reported by
 *           tm_poll_error as TM_ERR_INVALID_ARG.  Groups must be contiguous
 *           in K (no activation-order row permutation).
 *   scales  device, [K/group][N] of type dtype
 * Shapes, alignment, groups and ownership as for tm_pack_w4. */
tm_status tm_pack_awq(const int32_t *qweight, const int32_t *qzeros, const void *scales, int K, int N,
                      int group, tm_dtype dtype, void *stream, tm_packed **out);
tm_status tm_pack_gptq(const int32_t *qweight, const int32_t *qzeros, const void *scales, int zero_offset,
                       int K, int N, int group, tm_dtype dtype, void *stream, tm_packed **out);

/* 8-bit weights on the same pipeline (TurboMind paper, arXiv abstract:
 * "hybrid precision formats"; pith.science review, Figure 12 legend: FP8
 * weights).  The pages print no format; read as the int4 method with 8-bit
 * codes, one rounding per weight:
 *   tm_pack_w8   W = T(s * (q - z)), q and z in 0..255; zeros device
 *                [K/group][N] bytes, or NULL for the symmetric format (z = 128)
 *   tm_pack_fp8  W = T(s * e4m3(q)): q are FP8 E4M3 ("fn": bias 7, no
 *                infinities) bit patterns; no zeros.  The NaN codes 0x7F and
 *                0xFF give NaN weights.
 *   q       device, [K][N] uint8 codes
 *   scales  device, [K/group][N] 16-bit values of type dtype
 * Packed layout: 128-column tiles, 64-K blocks of 8192 bytes; inside a block
 * 16-byte chunk kq * 128 + c holds the 16 consecutive K values 16 kq + 0..15
 * of column c.  Zeros are tile-major [N/128][K/G][128] bytes.  Shapes, groups,
 * alignment and ownership as for tm_pack_w4.  These weights run on the
 * CUDA-core GEMV (M <= 8), the DECODE_MMA kernel (M <= 16, groups of at
 * least 64, dq_warps 1, 2, 4 or 8) and the TC kernel (any M); the other
 * kernels and dq_warps 16 report TM_ERR_UNSUPPORTED for them. */
tm_status tm_pack_w8(const uint8_t *q, const void *scales, const uint8_t *zeros, int K, int N, int group,
                     tm_dtype dtype, void *stream, tm_packed **out);
tm_status tm_pack_fp8(const uint8_t *q, const void *scales, int K, int N, int group, tm_dtype dtype,
                      void *stream, tm_packed **out);

/* Online GEMM (TurboMind paper, arXiv abstract: the online half of the pipeline;
 * pith.science review, Figure 9: dequantization overlapped with the MMA).
 *   A  device, [M][K] values of the handle's dtype, 16-byte aligned
 *   W  packed weight from tm_pack_w4 with matching K and N
 *   C  device, [M][N] output of the handle's dtype (caller-allocated),
 *      16-byte aligned; fp32 accumulation, one round-to-nearest-even at
 *      the end.  Results do not depend on the split or launch order.
 *   M == 0 is a no-op.  M <= 65535*256.
 *   Uses a library-owned split-K workspace per (device, stream), grown on
 *   demand; a call that would need to grow it while `stream` is being
 *   captured into a CUDA graph returns TM_ERR_UNSUPPORTED -- make one call
 *   of the same shape outside capture first.  Calls on the same stream are
 *   ordered; calls on different streams use different workspaces. */
tm_status tm_gemm_w4a16(const void *A, const tm_packed *W, void *C, int M, int N, int K,
                        void *stream);

/* As tm_gemm_w4a16 with an explicit kernel variant (cfg != NULL); used by
 * the tuner, the tests and the benchmark.  TM_ERR_UNSUPPORTED if the
 * variant cannot run this shape. */
tm_status tm_gemm_w4a16_ex(const void *A, const tm_packed *W, void *C, int M, int N, int K,
                           const tm_config *cfg, void *stream);

/* As tm_gemm_w4a16, for callers that cannot allocate device memory: an
 * application that owns all GPU memory through its own pool allocator and
 * forbids allocations behind its back.  The paper has no counterpart; this
 * is a deployment variant of the same GEMM.
 *   Allocates nothing: no cudaMalloc/cudaFree and no allocating library
 *   call.  Split-K partials and arrival counters live in static device
 *   arrays of the library (8 MiB of partials and 16384 counters, held on
 *   every GPU that loads the library until the process exits); a shape
 *   whose selected variant needs more returns TM_ERR_UNSUPPORTED with the
 *   sizes in tm_last_error().
 *   The first call on a device looks up the arrays' device addresses
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   All calls share one scratch per device and it keeps the last call's
 *   contents: calls that overlap on the GPU (different streams, or
 *   different host threads) race and give wrong results; order them.
 *   Each call clears the counters it uses with cudaMemsetAsync on `stream`.
 *   A bounded wait that gives up is recorded in a static device word of
 *   its own, which tm_poll_error reads and clears together with the
 *   regular error word (C of that call is then undefined). */
tm_status tm_gemm_w4a16_noalloc(const void *A, const tm_packed *W, void *C, int M, int N, int K,
                                void *stream);

/* Dequant-only (TurboMind paper, pith.science review, Figure 6: the runtime
 * conversion of the packed integers to floating point, then the scaling):
 *   W_out  device, [K][N] of the handle's dtype, 16-byte aligned, caller-
 *          allocated; W_out[k][n] = T(s[k/G][n] * (q[k][n] - z[k/G][n])),
 *          bit-exact with a single round-to-nearest-even per element (for
 *          8-bit handles the 8-bit formula of tm_pack_w8 / tm_pack_fp8).
 * Stream-ordered on `stream`; TM_ERR_INVALID_ARG for a bad handle or a
 * misaligned / NULL W_out. */
tm_status tm_dequant_w4(const tm_packed *W, void *W_out, void *stream);

/* Releases a packed weight (stream-ordered cudaFreeAsync). NULL is OK. */
tm_status tm_packed_free(tm_packed *W, void *stream);

/* Fills *info (host) with the handle's shape and device pointers. */
tm_status tm_packed_get(const tm_packed *W, tm_packed_info *info);

/* The variant tm_gemm_w4a16 would run for this handle and M (host only):
 * the environment override TM_VARIANT="kernel:block_m:split_k:dq_warps"
 * (kernel gemv, tc, tc_decode, decode_mma or its number) when it can run
 * this shape, else the tuned table's entry for M's row bucket, else the
 * built-in rule, set from crossovers measured on GB300: up to 4 rows and at
 * most 16 MB of packed weight, the register-MMA decode kernel in clusters
 * of 8 CTAs per tile; up to 8 rows its persistent stream-K grid; up to 64
 * rows the tcgen05 decode kernel; beyond, the tcgen05 kernel (groups of 32:
 * the CUDA-core GEMV up to 8 rows, else the tcgen05 kernel; 8-bit weights:
 * the CUDA-core GEMV up to 8 rows, the register-MMA decode kernel up to 16,
 * else the tcgen05 kernel). */
tm_status tm_select(const tm_packed *W, int M, tm_config *out);

/* Variant selection by measured throughput (the pages give no selection
 * rule; it follows from the measured crossovers between the kernels).  For
 * each M in Ms[0..nM), times every legal variant on `stream` (synchronises
 * it) the way applications run them: a CUDA graph of back-to-back launches
 * (programmatic dependent launch on) over rotated copies of the weight, so
 * that no launch finds its weights in L2; the median of three replays.  The
 * built-in choice is measured first and a later variant replaces the best so
 * far only if it is at least 2% faster, which keeps picks stable under
 * timing noise.  The winner is recorded in the process-wide table used by
 * tm_gemm_w4a16 under the key (N, K, group, dtype, symmetric, row bucket),
 * the row bucket being the next power of two >= M.  If the environment
 * variable TM_TUNE_CACHE names a file, the table is saved there.  best_out
 * (host, may be NULL) receives nM configs.  Allocates temporary device
 * copies of the weight (at most 7 besides W) and frees them before
 * returning.
 * Deviation from the plain tm_tune(Ms, W, stream) signature: best_out. */
tm_status tm_tune(const int *Ms, int nM, const tm_packed *W, void *stream, tm_config *best_out);

/* Pipeline geometry of the tcgen05 variant (block_m, dq_warps); host only,
 * needs no GPU.  *stages: shared-memory stages; *kblocks_per_stage: 64-K
 * blocks per stage; *tmem_slots: TMEM slots for dequantized 64-K blocks;
 * *legal: 1 if the variant can run, 0 if it is refused because some of its
 * mbarrier parity waits could start two phases ahead (the pages give no
 * pipeline; this is the Blackwell restatement of the overlap of pith.science
 * review Figure 9). */
tm_status tm_tc_pipeline(int block_m, int dq_warps, int *stages, int *kblocks_per_stage,
                         int *tmem_slots, int *legal);

/* Pipeline geometry of the TM_KERNEL_TC_DECODE kernel for (block_m,
 * dq_warps): the depth of its weight-stage ring (stages of four 64-K blocks;
 * a multiple of the warpgroup count, so a slot always feeds one
 * warpgroup), the activation stages and TMEM operand slots each warpgroup
 * owns, and whether the variant is accepted.  Host-only; for tests and
 * tools.  Returns TM_ERR_INVALID_ARG on NULL outputs. */
tm_status tm_tc_decode_pipeline(int block_m, int dq_warps, int *weight_stages,
                                int *act_stages_per_wg, int *tmem_slots_per_wg, int *legal);

/* Stream-K plan of the TM_KERNEL_TC_DECODE kernel for an M x N x K GEMM on a
 * GPU with `sm_count` SMs: the persistent grid (CTAs), the number of output
 * tiles (128 weight columns x block_m rows) and the fp32 partial slots per
 * tile that the split fix-up needs (1: no tile is cut between CTAs, no
 * scratch).  CTA c owns the (tile, 256-K stage) units [c*U/grid,
 * (c+1)*U/grid) of the U = tiles * ceil(K/256) units.  Host-only.
 * Returns TM_ERR_INVALID_ARG for sizes the GEMM would reject. */
tm_status tm_decode_plan(int M, int N, int K, int block_m, int sm_count, int *grid,
                         long long *tiles, int *partial_slots);

/* Decode attention over a low-bit KV cache: one query token per sequence
 * against its cached keys and values (TurboMind paper, pith.science review,
 * Figure 4: the attention pipeline dequantizes the low-bit cache by
 * integer-to-float conversion and scaling, then computes Q K^T and P V;
 * Figure 10: the cache is consumed in 64-token tiles).  For sequence b and
 * query head hq, with KV head h = hq / (Hq / Hkv) and t < lens[b]:
 *   K[t][d] = T(k_scale[t] * (kq[t][d] - k_zero[t])), V likewise
 *   O[b][hq] = sum_t softmax_t(sm_scale * Q[b][hq] . K[t]) V[t]
 * (per-token, per-KV-head scale and integer zero; one round-to-nearest-even
 * per cached element, as for the weights).  A sequence with lens[b] == 0
 * gets O = 0.
 *   q        device, [B][Hq][128] of dtype
 *   k_cache, v_cache  device, [B][Hkv][L_max][128 * kv_bits / 8] bytes;
 *            8 bits: one code 0..255 per byte; 4 bits: element d in byte
 *            d / 2, the low nibble holding even d
 *   k_scale, v_scale  device, [B][Hkv][L_max] of dtype
 *   k_zero, v_zero    device, [B][Hkv][L_max] bytes (codes; <= 15 for 4 bits)
 *   lens     device, [B] int32 (values outside [0, L_max] are clamped)
 *   o        device, [B][Hq][128] of dtype, written
 *   head_dim must be 128; Hq a multiple of Hkv with at most 16 query heads
 *   per KV head; L_max a positive multiple of 64; B * Hkv * L_max < 2^31;
 *   every pointer 16-byte aligned.  Cache rows at t >= lens[b] are never
 *   used (they may hold anything, NaN scales included).
 *   chunk_tiles: 64-token tiles per unit of work (0 = chosen from the
 *   shapes; tm_attn_decode_plan reports the choice).  Sequences longer
 *   than one unit are split over CTAs and merged through a library-owned
 *   per-(device, stream) workspace (grown outside stream capture, like the
 *   GEMM's split-K scratch).
 * The caller owns every buffer.  Stream-ordered on `stream`, launched with
 * programmatic dependent launch like the GEMMs (every read of the inputs
 * waits for the previous kernel).  Device-side conditions (a bounded wait
 * that gave up) are reported by tm_poll_error.  TM_ERR_INVALID_ARG /
 * TM_ERR_UNSUPPORTED for arguments outside the above. */
tm_status tm_attn_decode(const void *q, const uint8_t *k_cache, const void *k_scale, const uint8_t *k_zero,
                         const uint8_t *v_cache, const void *v_scale, const uint8_t *v_zero, const int32_t *lens,
                         void *o, int B, int Hq, int Hkv, int head_dim, int L_max, int kv_bits, tm_dtype dtype,
                         float sm_scale, int chunk_tiles, void *stream);

/* The automatic chunk_tiles of tm_attn_decode and its grid (CTAs) for the
 * shape on the current device, host-side (planned for every sequence at
 * L_max).  TM_ERR_INVALID_ARG for shapes tm_attn_decode refuses. */
tm_status tm_attn_decode_plan(int B, int Hq, int Hkv, int L_max, int kv_bits, tm_dtype dtype, int *chunk_tiles,
                              int *grid);

/* Loads/saves the tuned table (JSON lines) from/to a host path. */
tm_status tm_tune_load(const char *path);
tm_status tm_tune_save(const char *path);

/* Synchronises `stream`, then reads and clears the current device's error
 * words (the regular one and the static one of tm_gemm_w4a16_noalloc):
 * TM_ERR_TIMEOUT if a bounded wait gave up, TM_ERR_INVALID_ARG if a code
 * byte was above 15, TM_OK otherwise.  Allocates nothing after the first
 * call on a device. */
tm_status tm_poll_error(void *stream);

/* Self-test of the bounded wait used by every kernel: launches one CTA
 * that waits on a barrier nothing will complete, with a limit of
 * `limit_ns` nanoseconds (1000..10^9).  The wait gives up, records
 * TM_ERR_TIMEOUT in the error word and the kernel returns normally; read
 * it with tm_poll_error. */
tm_status tm_selftest_wait_timeout(long long limit_ns, void *stream);

/* Message for the calling thread's last non-OK status ("" if none). */
const char *tm_last_error(void);

/* Library version string. */
const char *tm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TMW4_H */

"""Oracle for weight-only int4 x fp16/bf16 GEMM (W4A16) -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA path.

What the method computes (TurboMind paper, arXiv abstract: a mixed-precision
matrix multiply whose weights are packed once offline and consumed by an
accelerated online kernel; pith.science review, Figure 6: runtime I2F
conversion and scaling of the packed low-bit values before the MMA):

    W[k, n] = RNE_T( s[g, n] * (q[k, n] - z[g, n]) ),   g = k // G
    C       = A @ W            (accumulated exactly here, in float64)

with q, z in [0, 15], s a 16-bit float of type T (fp16 or bf16) and A an
[M, K] matrix of type T.  The product s*(q-z) is exact in float64 (s has at
most 11 significant bits, |q-z| at most 4), so RNE_T is the single rounding
of the exact real product.

Readings taken where the pages are silent:
  * logical weight W is [K, N], C = A @ W with A [M, K] and C [M, N], both
    row-major; scales/zeros are [K/G, N];
  * symmetric quantization has no stored zero and uses z = 8;
  * the packed layout is this library's own (the pages' Ampere fragment
    order is prior art); ``pack_ref``/``unpack_ref`` below are written from
    the layout specification, not from any kernel source.

Parity status: every function here is pinned by CPU tests against closed
forms, exact rational arithmetic, brute force or fixed bit patterns (see
tests/test_oracle_*.py).  No function is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# 16-bit float encodings
# ---------------------------------------------------------------------------


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16) -> exact float64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values.

    bfloat16 is the upper half of an IEEE binary32 word, so widening is a
    16-bit left shift of the pattern.
    """
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def rne_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to binary16, round-to-nearest-even; return bits.

    numpy converts float64 -> float16 with correct IEEE rounding (nearest,
    ties to even, gradual underflow).  The CPU tests pin this against exact
    rational rounding and fixed bit patterns.
    """
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def rne_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16, round-to-nearest-even; return bits.

    Requires every finite input below 2^128 in magnitude to be exactly
    representable in binary32 (true for the dequant products here, which need
    at most 15 significant bits); larger magnitudes round to infinity.  The
    rounding is done on the binary32 pattern u: add 0x7FFF plus the lowest
    kept bit, then drop the low 16 bits; NaNs map to a quiet NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    huge = np.abs(x) >= 2.0 ** 128          # beyond binary32: rounds to infinity
    with np.errstate(over="ignore"):
        f32 = np.where(huge, np.copysign(np.inf, x), x).astype(np.float32)
    if not np.array_equal(np.where(huge, f32, f32.astype(np.float64)),
                          np.where(huge, f32, x), equal_nan=True):
        raise ValueError("rne_bf16_bits: input not exactly representable in binary32")
    u = f32.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint32)
    nan = np.isnan(f32)
    r = np.where(nan, (f32.view(np.uint32) >> np.uint32(16)) | np.uint32(0x0040), r)
    return r.astype(np.uint16)


def act_bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Activation / scale bit patterns of type ``dtype`` ('f16'|'bf16') -> float64."""
    if dtype == "f16":
        return f16_bits_to_f64(bits)
    if dtype == "bf16":
        return bf16_bits_to_f64(bits)
    raise ValueError(dtype)


def _rne_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return rne_f16_bits(x)
    if dtype == "bf16":
        return rne_bf16_bits(x)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# Dequantization (pith.science review, Figure 6: runtime I2F conversion and
# scaling; Figure 4 text: "I2F scaling" of low-bit values to FP16)
# ---------------------------------------------------------------------------


def _expand_groups(a: np.ndarray, group: int) -> np.ndarray:
    """[K/G, N] -> [K, N] by repeating each group row G times."""
    return np.repeat(a, group, axis=0)


def dequant_f64(q, scale_bits, zeros, group: int, dtype: str) -> np.ndarray:
    """Exact real products s*(q - z) as float64 (before rounding to T).

    q: [K, N] uint8 in 0..15.  scale_bits: [K/G, N] uint16 patterns of type
    ``dtype``.  zeros: [K/G, N] uint8 in 0..15, or None for the symmetric
    format (implicit zero 8).
    """
    q = np.asarray(q)
    K, N = q.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    s = act_bits_to_f64(scale_bits, dtype)
    if s.shape != (K // group, N):
        raise ValueError("scale shape mismatch")
    if zeros is None:
        z = np.full((K // group, N), 8, dtype=np.int64)
    else:
        z = np.asarray(zeros).astype(np.int64)
        if z.shape != (K // group, N):
            raise ValueError("zero shape mismatch")
    diff = q.astype(np.int64) - _expand_groups(z, group)
    return _expand_groups(s, group) * diff.astype(np.float64)


def dequant_bits(q, scale_bits, zeros, group: int, dtype: str) -> np.ndarray:
    """W = RNE_T(s * (q - z)) as uint16 bit patterns, shape [K, N]."""
    return _rne_bits(dequant_f64(q, scale_bits, zeros, group, dtype), dtype)


# ---------------------------------------------------------------------------
# GEMM (the plain definition, accumulated in float64)
# ---------------------------------------------------------------------------


def gemm_ref(a_bits, w_bits, dtype: str) -> np.ndarray:
    """C_ref = A @ W in float64 from the 16-bit patterns of A [M,K] and W [K,N].

    Each product a*w is exact in float64 (at most 11+11 significant bits);
    the K-sum rounding (<= K * 2^-53 * sum|a*w|) is negligible against the
    GEMM tolerance.  C_ref is not rounded to 16 bits.
    """
    A = act_bits_to_f64(a_bits, dtype)
    W = act_bits_to_f64(w_bits, dtype)
    return A @ W


def rms(c_ref: np.ndarray) -> float:
    """Root mean square over all elements of one problem's C_ref."""
    c = np.asarray(c_ref, dtype=np.float64)
    return float(np.sqrt(np.mean(c * c))) if c.size else 0.0


def max_err_ratio(c, c_ref, rms_value: float | None = None, rel: float = 1e-2) -> float:
    """max over elements of |C - C_ref| / (rel * (|C_ref| + rms(C_ref)))."""
    c = np.asarray(c, dtype=np.float64)
    c_ref = np.asarray(c_ref, dtype=np.float64)
    if c.size == 0:
        return 0.0
    r = rms(c_ref) if rms_value is None else rms_value
    bound = rel * (np.abs(c_ref) + r)
    err = np.abs(c - c_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                         np.where(err > 0, np.inf, 0.0))
    return float(np.max(ratio))


def tolerance_ok(c, c_ref, rms_value: float | None = None, rel: float = 1e-2) -> bool:
    """Per-element check |C - C_ref| <= rel * (|C_ref| + rms(C_ref))."""
    return max_err_ratio(c, c_ref, rms_value, rel) <= 1.0


# ---------------------------------------------------------------------------
# Packed layout reader/writer (the library's own Blackwell layout).
#
# The pages' packing (pith.science review, Figures 6 and 7) permutes each
# thread's eight 4-bit values so that after I2F they sit where the MMA wants
# them, and stores them in the order the runtime loads them, so that the
# online kernel needs no rearrangement.  Figures 23/24 print the in-register
# order of eight values in a 32-bit word: e7 e5 e3 e1 e6 e4 e2 e0 (high to
# low nibble): even elements in the low half-word, odd in the high half, so
# one mask yields two 16-bit lanes.  This library keeps that word order and
# defines its own tile order for its tcgen05 and GEMV consumers:
#
#   * K is a multiple of 64 and N of 128.  Columns form 128-wide tiles; tile
#     nt, K-block kb (64 values of K) is a 4096-byte block at byte
#     (nt * (K/64) + kb) * 4096, so all K of a tile is contiguous.
#   * A block holds two 2048-byte atoms, a = 0 for columns [0, 64) of the
#     tile and a = 1 for [64, 128).  An atom holds 512 little-endian 32-bit
#     words; word h*256 + nl*4 + j (h in {0,1}, nl in [0,64), j in [0,4))
#     holds the eight values q[64kb + 8o + e, 128nt + 64a + nl], e = 0..7,
#     with o = 4h + j.
#   * Value e sits at bits [4p, 4p+4) with p = NIBBLE_POS[e].
#   * Scales are reordered tile-major: [N/128][K/G][128] 16-bit patterns,
#     i.e. scale (g, n) at index (n//128 * (K/G) + g) * 128 + n%128.
#   * Zeros are nibble-packed, tile-major: [N/128][K/G][64] bytes; byte
#     (nt, g, i) holds column 128nt + 2i in the low nibble and 128nt + 2i + 1
#     in the high nibble.  The symmetric format stores no zeros.
# ---------------------------------------------------------------------------

TILE_N = 128
ATOM_K = 64
ATOM_N = 64
#: nibble position of element e (0..7) inside its 32-bit word
NIBBLE_POS = (0, 4, 1, 5, 2, 6, 3, 7)


def _atom_word_coords(K: int, N: int):
    """For every 32-bit word of the packed stream, (k0, n) of its first value.

    Returns two int64 arrays of length K*N/8 in packed-word order.
    """
    if K % ATOM_K or N % TILE_N:
        raise ValueError("K must be a multiple of 64 and N of 128")
    nkb = K // ATOM_K
    w = np.arange(K * N // 8, dtype=np.int64)
    block, inblk = w // 1024, w % 1024
    nt, kb = block // nkb, block % nkb
    a, widx = inblk // 512, inblk % 512
    h, rem = widx // 256, widx % 256
    nl, j = rem // 4, rem % 4
    o = 4 * h + j
    k0 = ATOM_K * kb + 8 * o
    n = TILE_N * nt + ATOM_N * a + nl
    return k0, n


def pack_ref(q: np.ndarray) -> np.ndarray:
    """q [K, N] uint8 (0..15) -> packed weight bytes (uint8, K*N/2)."""
    q = np.asarray(q)
    if q.dtype != np.uint8 or q.ndim != 2:
        raise ValueError("q must be a 2-D uint8 array")
    if np.any(q > 15):
        raise ValueError("q values must be in 0..15")
    K, N = q.shape
    k0, n = _atom_word_coords(K, N)
    words = np.zeros(k0.shape, dtype=np.uint32)
    for e in range(8):
        words |= q[k0 + e, n].astype(np.uint32) << np.uint32(4 * NIBBLE_POS[e])
    return words.astype("<u4").view(np.uint8)


def unpack_ref(packed: np.ndarray, K: int, N: int) -> np.ndarray:
    """Packed weight bytes -> q [K, N] uint8 (inverse of ``pack_ref``)."""
    b = np.ascontiguousarray(np.asarray(packed, dtype=np.uint8))
    if b.size != K * N // 2:
        raise ValueError("packed size mismatch")
    words = b.view("<u4").astype(np.uint32)
    k0, n = _atom_word_coords(K, N)
    q = np.zeros((K, N), dtype=np.uint8)
    for e in range(8):
        q[k0 + e, n] = (words >> np.uint32(4 * NIBBLE_POS[e])) & np.uint32(0xF)
    return q


def pack_scales_ref(scales: np.ndarray) -> np.ndarray:
    """scales [K/G, N] (16-bit patterns) -> tile-major [N/128, K/G, 128] (flattened)."""
    s = np.asarray(scales, dtype=np.uint16)
    G_rows, N = s.shape
    if N % TILE_N:
        raise ValueError("N must be a multiple of 128")
    return s.reshape(G_rows, N // TILE_N, TILE_N).transpose(1, 0, 2).reshape(-1).copy()


def unpack_scales_ref(sp: np.ndarray, G_rows: int, N: int) -> np.ndarray:
    """Inverse of ``pack_scales_ref``."""
    sp = np.asarray(sp, dtype=np.uint16).reshape(N // TILE_N, G_rows, TILE_N)
    return sp.transpose(1, 0, 2).reshape(G_rows, N).copy()


def pack_zeros_ref(zeros: np.ndarray) -> np.ndarray:
    """zeros [K/G, N] uint8 (0..15) -> tile-major nibble bytes [N/128, K/G, 64] (flattened)."""
    z = np.asarray(zeros, dtype=np.uint8)
    G_rows, N = z.shape
    if N % TILE_N:
        raise ValueError("N must be a multiple of 128")
    pairs = (z[:, 0::2] & 0xF) | ((z[:, 1::2] & 0xF) << 4)          # [K/G, N/2]
    return pairs.reshape(G_rows, N // TILE_N, TILE_N // 2).transpose(1, 0, 2).reshape(-1).copy()


def unpack_zeros_ref(zp: np.ndarray, G_rows: int, N: int) -> np.ndarray:
    """Inverse of ``pack_zeros_ref``."""
    zp = np.asarray(zp, dtype=np.uint8).reshape(N // TILE_N, G_rows, TILE_N // 2)
    pairs = zp.transpose(1, 0, 2).reshape(G_rows, N // 2)
    z = np.empty((G_rows, N), dtype=np.uint8)
    z[:, 0::2] = pairs & 0xF
    z[:, 1::2] = pairs >> 4
    return z

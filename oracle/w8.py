"""Oracle for 8-bit weights (W8A16: int8 codes with a zero point, and FP8
E4M3 codes) -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA path.

The pages name 8-bit weights among TurboMind's hybrid-precision formats
(TurboMind paper, arXiv abstract: "hybrid precision formats"; pith.science
review, Figure 12 legend: FP8 Qwen3 runs) but print no format.  Read as the
int4 method with 8-bit codes:

    int8:  W[k, n] = RNE_T( s[g, n] * (q[k, n] - z[g, n]) ),  q, z in 0..255
           (symmetric: no stored zero, z = 128)
    FP8:   W[k, n] = RNE_T( s[g, n] * e4m3(q[k, n]) ),         g = k // G

with e4m3 the OCP FP8 E4M3 ("fn") decoding: sign, 4 exponent bits with bias
7, 3 mantissa bits, exponent 0 subnormal, S.1111.111 NaN, no infinities.  The
products are exact in float64 (at most 20 significant bits), so RNE_T is the
single rounding of the exact real product, as for int4.

Packed 8-bit layout (the library's own): 128-column tiles, 64-K blocks of
8192 bytes at (nt * K/64 + kb) * 8192; inside a block, 16-byte chunk
kq * 128 + c holds the 16 consecutive K values 64 kb + 16 kq + (0..15) of
column 128 nt + c, byte e being K offset e.  Zeros are bytes, tile-major
[N/128][K/G][128]; scales as for int4.

Parity: pinned by tests/test_oracle_w8.py (torch's independent FP8 decoder,
q - z = +-1 giving the scale itself, chunk and block properties of the
layout, round trips).
"""

from __future__ import annotations

import numpy as np

from .w4a16 import _rne_bits, act_bits_to_f64, TILE_N, ATOM_K


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """FP8 E4M3 (fn) bit patterns (uint8) -> exact float64 values (NaN codes -> nan)."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    sub = m * 2.0 ** -9
    norm = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    v = sign * np.where(e == 0, sub, norm)
    return np.where((e == 15) & ((b & 7) == 7), np.nan, v)


def _expand(a: np.ndarray, group: int) -> np.ndarray:
    return np.repeat(a, group, axis=0)


def dequant8_f64(q, scale_bits, zeros, group: int, dtype: str, fp8: bool = False) -> np.ndarray:
    """Exact products (before rounding to T) for 8-bit codes q [K, N] uint8."""
    q = np.asarray(q, dtype=np.uint8)
    K, N = q.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    s = act_bits_to_f64(scale_bits, dtype)
    if s.shape != (K // group, N):
        raise ValueError("scale shape mismatch")
    if fp8:
        if zeros is not None:
            raise ValueError("FP8 codes have no zero point")
        return _expand(s, group) * e4m3_to_f64(q)
    z = np.full((K // group, N), 128, dtype=np.int64) if zeros is None else np.asarray(zeros).astype(np.int64)
    if z.shape != (K // group, N):
        raise ValueError("zero shape mismatch")
    return _expand(s, group) * (q.astype(np.int64) - _expand(z, group)).astype(np.float64)


def dequant8_bits(q, scale_bits, zeros, group: int, dtype: str, fp8: bool = False) -> np.ndarray:
    """W as uint16 bit patterns of type ``dtype``, shape [K, N]."""
    return _rne_bits(dequant8_f64(q, scale_bits, zeros, group, dtype, fp8), dtype)


def _chunk_coords(K: int, N: int):
    """(k0, n) of every 16-byte chunk of the packed 8-bit stream, in stream order."""
    if K % ATOM_K or N % TILE_N:
        raise ValueError("K must be a multiple of 64 and N of 128")
    nkb = K // ATOM_K
    c = np.arange(K * N // 16, dtype=np.int64)
    block, inblk = c // 512, c % 512
    nt, kb = block // nkb, block % nkb
    kq, col = inblk // TILE_N, inblk % TILE_N
    return ATOM_K * kb + 16 * kq, TILE_N * nt + col


def pack8_ref(q: np.ndarray) -> np.ndarray:
    """q [K, N] uint8 codes -> packed bytes (K * N)."""
    q = np.asarray(q, dtype=np.uint8)
    K, N = q.shape
    k0, n = _chunk_coords(K, N)
    out = np.zeros((k0.size, 16), dtype=np.uint8)
    for e in range(16):
        out[:, e] = q[k0 + e, n]
    return out.reshape(-1)


def unpack8_ref(packed: np.ndarray, K: int, N: int) -> np.ndarray:
    """Inverse of ``pack8_ref``."""
    b = np.asarray(packed, dtype=np.uint8).reshape(-1, 16)
    k0, n = _chunk_coords(K, N)
    q = np.zeros((K, N), dtype=np.uint8)
    for e in range(16):
        q[k0 + e, n] = b[:, e]
    return q


def pack_zeros8_ref(zeros: np.ndarray) -> np.ndarray:
    """zeros [K/G, N] uint8 -> tile-major bytes [N/128, K/G, 128] (flattened)."""
    z = np.asarray(zeros, dtype=np.uint8)
    G_rows, N = z.shape
    return z.reshape(G_rows, N // TILE_N, TILE_N).transpose(1, 0, 2).reshape(-1).copy()

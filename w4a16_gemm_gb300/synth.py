"""Seeded synthetic inputs for the W4A16 GEMM (shared by tests and bench).

This module draws the random weights and activations and turns the weights
into int4 codes with a round-to-nearest (RTN) quantizer.  The quantizer is the
stand-in for the AWQ/GPTQ checkpoints the source pages evaluate with (their
models are "Qwen3 8B AWQ" and similar): it produces the *inputs* of the
method -- codes q, scales s and zeros z -- and is not part of the method's own
arithmetic (packing, dequantization, multiply).  Nothing here imports the
CUDA library or the oracle.

Workloads (8B-class decoder layer: hidden 4096, FFN 14336; 70B-class layer:
hidden 8192, FFN 28672; weights drawn N(0, 0.02) in fp32 before
quantization):

  tiny         K=256,  N=256,  M=1,            asym G=128, fp16
  decode_8b    4 shapes,       M in {1,4,16},   asym G=128, fp16
  prefill_8b   4 shapes,       M in {512,2048,8192}, asym G=128, bf16
  class_70b    4 shapes,       M in {1,64,4096}, asym G=128, fp16
  sym_g64      2 shapes,       M in {1,2,8,32,128,512,2048,8192},
               symmetric G=64 (z = 8), Student-t(3)*0.5 activations
               clipped to +-64, fp16

Seeds: the tiny problem draws weights then activations from
``default_rng(0)``; every other problem draws its weights in chunks of
CHUNK_ROWS rows of K, chunk j from ``default_rng(SeedSequence([cfg, shape, 0,
j]))`` (a multiple of every group size, so quantization groups never straddle
chunks), and the activations for row count M in chunks of CHUNK_ROWS rows of
M, chunk j from ``default_rng(SeedSequence([cfg, shape, 1, M, j]))``.  The
chunks are independent streams, drawn in parallel threads.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
from dataclasses import dataclass

import numpy as np

CHUNK_ROWS = 1024


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:
        return max(1, min(16, os.cpu_count() or 1))


def _chunked(rows: int, fn) -> np.ndarray:
    """Concatenates fn(j, r0, r1) over row chunks [r0, r1) of CHUNK_ROWS rows,
    computed in parallel threads (numpy releases the GIL in the heavy work)."""
    bounds = [(j, r0, min(rows, r0 + CHUNK_ROWS)) for j, r0 in enumerate(range(0, rows, CHUNK_ROWS))]
    if len(bounds) == 1:
        return fn(*bounds[0])
    with cf.ThreadPoolExecutor(max_workers=_threads()) as ex:
        parts = list(ex.map(lambda b: fn(*b), bounds))
    return parts

SHAPES_8B = ((4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096))
SHAPES_70B = ((8192, 10240), (8192, 8192), (8192, 57344), (28672, 8192))
SHAPES_SYM = ((5120, 34816), (17408, 5120))


@dataclass(frozen=True)
class Workload:
    """One named synthetic workload: its shapes, row counts and format."""

    name: str
    cfg_id: int
    shapes: tuple
    ms: tuple
    dtype: str          # 'f16' or 'bf16' (activations, scales and output)
    group: int
    symmetric: bool
    act_dist: str       # 'normal' or 'student_t3'


WORKLOADS = {
    "tiny": Workload("tiny", 0, ((256, 256),), (1,), "f16", 128, False, "normal"),
    "decode_8b": Workload("decode_8b", 1, SHAPES_8B, (1, 4, 16), "f16", 128, False, "normal"),
    "prefill_8b": Workload("prefill_8b", 2, SHAPES_8B, (512, 2048, 8192), "bf16", 128, False,
                           "normal"),
    "class_70b": Workload("class_70b", 3, SHAPES_70B, (1, 64, 4096), "f16", 128, False, "normal"),
    "sym_g64": Workload("sym_g64", 4, SHAPES_SYM, (1, 2, 8, 32, 128, 512, 2048, 8192), "f16", 64,
                        True, "student_t3"),
}


@dataclass
class QuantWeight:
    """Quantized weight: codes q [K,N] u8, scale bit patterns [K/G,N] u16,
    zeros [K/G,N] u8 (None for the symmetric format)."""

    q: np.ndarray
    scales: np.ndarray
    zeros: np.ndarray | None
    group: int
    dtype: str

    @property
    def K(self) -> int:
        return self.q.shape[0]

    @property
    def N(self) -> int:
        return self.q.shape[1]


def to_16bit(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32/fp64 array -> 16-bit patterns of ``dtype`` (uint16), RNE."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch  # float32 -> bfloat16 conversion (round to nearest even)

        t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(dtype)


def from_16bit_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit patterns -> float32 values (exact widening)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_rtn(w: np.ndarray, group: int, dtype: str, symmetric: bool) -> QuantWeight:
    """Group-wise RTN int4 quantization of an fp32 weight [K, N].

    Asymmetric: per column and K-group, s = T((max-min)/15),
    z = clamp(rint(-min/s), 0, 15), q = clamp(rint(x/s) + z, 0, 15).
    Symmetric: s = T(max|x|/7), q = clamp(rint(x/s) + 8, 0, 15).
    The division uses the stored (rounded) scale; rint is round-half-even in
    fp32.  A group whose scale rounds to zero stores s = 0, z = 0, q = 0.
    """
    w = np.asarray(w, dtype=np.float32)
    K, N = w.shape
    if K % group:
        raise ValueError("K must be a multiple of group")
    g = w.reshape(K // group, group, N)
    if symmetric:
        amax = np.max(np.abs(g), axis=1)
        s_bits = to_16bit(amax / np.float32(7.0), dtype)
    else:
        mn = np.min(g, axis=1)
        mx = np.max(g, axis=1)
        s_bits = to_16bit((mx - mn) / np.float32(15.0), dtype)
    s = from_16bit_f32(s_bits, dtype)
    dead = s == 0
    s_safe = np.where(dead, np.float32(1.0), s).astype(np.float32)
    if symmetric:
        z = None
        zq = np.float32(8.0)
        qf = np.rint(g / s_safe[:, None, :]) + zq
    else:
        zf = np.clip(np.rint(-mn / s_safe), 0, 15).astype(np.float32)
        zf = np.where(dead, np.float32(0.0), zf)
        z = zf.astype(np.uint8)
        qf = np.rint(g / s_safe[:, None, :]) + zf[:, None, :]
    q = np.clip(qf, 0, 15)
    q = np.where(dead[:, None, :], np.float32(0.0), q).astype(np.uint8)
    return QuantWeight(q.reshape(K, N), s_bits, z, group, dtype)


def _draw_acts(rng: np.random.Generator, M: int, K: int, dist: str, dtype: str) -> np.ndarray:
    if dist == "normal":
        a = rng.standard_normal((M, K), dtype=np.float32)
    elif dist == "student_t3":
        a = np.clip(0.5 * rng.standard_t(3, size=(M, K)), -64.0, 64.0).astype(np.float32)
    else:
        raise ValueError(dist)
    return to_16bit(a, dtype)


def weight(workload: str, shape_idx: int) -> QuantWeight:
    """Quantized weight of one shape of a named workload."""
    wl = WORKLOADS[workload]
    K, N = wl.shapes[shape_idx]
    if wl.cfg_id == 0:
        rng = np.random.default_rng(0)
        w = rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.02)
        return quantize_rtn(w, wl.group, wl.dtype, wl.symmetric)

    def chunk(j, r0, r1):
        rng = np.random.default_rng(np.random.SeedSequence([wl.cfg_id, shape_idx, 0, j]))
        w = rng.standard_normal((r1 - r0, N), dtype=np.float32) * np.float32(0.02)
        return quantize_rtn(w, wl.group, wl.dtype, wl.symmetric)

    parts = _chunked(K, chunk)
    if isinstance(parts, QuantWeight):
        return parts
    return QuantWeight(np.concatenate([q.q for q in parts]), np.concatenate([q.scales for q in parts]),
                       None if wl.symmetric else np.concatenate([q.zeros for q in parts]),
                       wl.group, wl.dtype)


def activations(workload: str, shape_idx: int, M: int) -> np.ndarray:
    """Activation bit patterns [M, K] (uint16) for one shape and row count."""
    wl = WORKLOADS[workload]
    K, N = wl.shapes[shape_idx]
    if wl.cfg_id == 0:
        rng = np.random.default_rng(0)
        rng.standard_normal((K, N), dtype=np.float32)  # weights come first
        return _draw_acts(rng, M, K, wl.act_dist, wl.dtype)

    def chunk(j, r0, r1):
        rng = np.random.default_rng(np.random.SeedSequence([wl.cfg_id, shape_idx, 1, M, j]))
        return _draw_acts(rng, r1 - r0, K, wl.act_dist, wl.dtype)

    parts = _chunked(M, chunk)
    return parts if isinstance(parts, np.ndarray) else np.concatenate(parts)


def random_problem(seed: int, M: int, K: int, N: int, group: int = 128, dtype: str = "f16",
                   symmetric: bool = False, act_dist: str = "normal"):
    """A free-form seeded problem (for tests at arbitrary sizes).

    Returns (QuantWeight, activation bits [M, K]).
    """
    rng = np.random.default_rng(np.random.SeedSequence([1000 + seed, M, K, N, group]))
    w = rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.02)
    qw = quantize_rtn(w, group, dtype, symmetric)
    a = _draw_acts(rng, M, K, act_dist, dtype)
    return qw, a


# ------------------------------------------------------------ decode attention
@dataclass
class KVProblem:
    """One decode-attention step over a low-bit KV cache (layouts as the
    library takes them): q [B, Hq, D] 16-bit patterns; codes [B, Hkv, L_max,
    D * bits / 8] bytes (4 bits: two elements per byte, low nibble first);
    scales [B, Hkv, L_max] 16-bit patterns; zeros [B, Hkv, L_max] bytes;
    lens [B] int32."""
    q: np.ndarray
    k_codes: np.ndarray
    k_scale: np.ndarray
    k_zero: np.ndarray
    v_codes: np.ndarray
    v_scale: np.ndarray
    v_zero: np.ndarray
    lens: np.ndarray
    bits: int
    dtype: str
    sm_scale: float

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def Hq(self) -> int:
        return self.q.shape[1]

    @property
    def D(self) -> int:
        return self.q.shape[2]

    @property
    def Hkv(self) -> int:
        return self.k_codes.shape[1]

    @property
    def L_max(self) -> int:
        return self.k_codes.shape[2]


def kv_problem(seed: int, B: int, Hq: int, Hkv: int, D: int, lens, L_max: int | None = None,
               bits: int = 8, dtype: str = "f16") -> KVProblem:
    """Seeded synthetic cache: N(0, 1) queries; uniform codes (4 bits: uniform
    bytes, i.e. two uniform nibbles) and zeros; per-token scales uniform in
    [0.004, 0.012] (8 bits) or [0.06, 0.2] (4 bits), so that K and V values
    span about +-2; sm_scale = 1 / sqrt(D)."""
    lens = np.asarray(lens, dtype=np.int32)
    if L_max is None:
        L_max = max(64, int(-(-int(lens.max(initial=0)) // 64) * 64))
    rng = np.random.default_rng(np.random.SeedSequence([7000 + seed, B, Hq, Hkv, D, L_max, bits]))
    q = to_16bit(rng.standard_normal((B, Hq, D), dtype=np.float32), dtype)
    width = D if bits == 8 else D // 2
    zhi = 256 if bits == 8 else 16
    lo, hi = (0.004, 0.012) if bits == 8 else (0.06, 0.2)

    def side():
        codes = rng.integers(0, 256, size=(B, Hkv, L_max, width), dtype=np.uint8)
        scale = to_16bit(rng.uniform(lo, hi, size=(B, Hkv, L_max)).astype(np.float32), dtype)
        zero = rng.integers(0, zhi, size=(B, Hkv, L_max), dtype=np.uint8)
        return codes, scale, zero

    kc, ks, kz = side()
    vc, vs, vz = side()
    return KVProblem(q, kc, ks, kz, vc, vs, vz, lens, bits, dtype, float(1.0 / np.sqrt(D)))


@dataclass(frozen=True)
class AttnWorkload:
    """Decode attention at an 8B-class head layout (32 query heads, 8 KV heads,
    head dim 128) for a list of (batch, context-length range) cases; lengths
    are drawn uniformly from the range per sequence."""
    bits: int
    dtype: str = "f16"
    Hq: int = 32
    Hkv: int = 8
    D: int = 128
    cases: tuple = ((1, (8192, 8192)), (16, (1024, 8192)), (64, (512, 4096)), (256, (256, 2048)))


ATTN_WORKLOADS = {
    "attn_8b_kv8": AttnWorkload(bits=8),
    "attn_8b_kv4": AttnWorkload(bits=4),
}


def attn_lens(name: str, case_idx: int) -> np.ndarray:
    wl = ATTN_WORKLOADS[name]
    B, (lo, hi) = wl.cases[case_idx]
    rng = np.random.default_rng(np.random.SeedSequence([7100, wl.bits, case_idx]))
    return rng.integers(lo, hi + 1, size=B).astype(np.int32)

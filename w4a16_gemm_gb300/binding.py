"""ctypes binding of libtmw4.so (argument marshalling only).

Every step of the W4A16 path runs in the library's CUDA kernels; this module
turns torch tensors into device pointers and the current CUDA stream into a
``cudaStream_t``, calls the C ABI declared in ``include/tmw4.h`` and raises
:class:`TmError` on a non-OK status.  There is no fallback: if the library is
missing, :func:`lib` raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtmw4.so")

TM_OK, TM_ERR_INVALID_ARG, TM_ERR_UNSUPPORTED, TM_ERR_CUDA, TM_ERR_OOM, TM_ERR_TIMEOUT = range(6)
TM_F16, TM_BF16 = 0, 1
TM_KERNEL_AUTO, TM_KERNEL_GEMV, TM_KERNEL_TC, TM_KERNEL_TC_DECODE, TM_KERNEL_DECODE_MMA = 0, 1, 2, 3, 4
STATUS_NAMES = {0: "TM_OK", 1: "TM_ERR_INVALID_ARG", 2: "TM_ERR_UNSUPPORTED", 3: "TM_ERR_CUDA",
                4: "TM_ERR_OOM", 5: "TM_ERR_TIMEOUT"}


class TmError(RuntimeError):
    """A non-OK tm_status, with the library's message."""

    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class TmConfig(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("block_m", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("dq_warps", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {"kernel": {1: "gemv", 2: "tc", 3: "tc_decode", 4: "decode_mma"}.get(self.kernel, self.kernel),
                "block_m": self.block_m, "split_k": self.split_k, "dq_warps": self.dq_warps}


class TmPackedInfo(ctypes.Structure):
    _fields_ = [("K", ctypes.c_int32), ("N", ctypes.c_int32), ("group", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("symmetric", ctypes.c_int32), ("device", ctypes.c_int32),
                ("qweight", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zeros", ctypes.c_void_p),
                ("qweight_bytes", ctypes.c_size_t), ("scales_bytes", ctypes.c_size_t),
                ("zeros_bytes", ctypes.c_size_t), ("bits", ctypes.c_int32), ("fp8", ctypes.c_int32)]


_LIB = None

#: (name, restype, argtypes) of every entry point in include/tmw4.h
_VP, _I, _LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
SIGNATURES = [
    ("tm_pack_w4", _I, [_VP, _VP, _VP, _I, _I, _I, _I, _VP, ctypes.POINTER(_VP)]),
    ("tm_pack_awq", _I, [_VP, _VP, _VP, _I, _I, _I, _I, _VP, ctypes.POINTER(_VP)]),
    ("tm_pack_w8", _I, [_VP, _VP, _VP, _I, _I, _I, _I, _VP, ctypes.POINTER(_VP)]),
    ("tm_pack_fp8", _I, [_VP, _VP, _I, _I, _I, _I, _VP, ctypes.POINTER(_VP)]),
    ("tm_pack_gptq", _I, [_VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, ctypes.POINTER(_VP)]),
    ("tm_gemm_w4a16", _I, [_VP, _VP, _VP, _I, _I, _I, _VP]),
    ("tm_gemm_w4a16_ex", _I, [_VP, _VP, _VP, _I, _I, _I, ctypes.POINTER(TmConfig), _VP]),
    ("tm_gemm_w4a16_noalloc", _I, [_VP, _VP, _VP, _I, _I, _I, _VP]),
    ("tm_dequant_w4", _I, [_VP, _VP, _VP]),
    ("tm_packed_free", _I, [_VP, _VP]),
    ("tm_packed_get", _I, [_VP, ctypes.POINTER(TmPackedInfo)]),
    ("tm_select", _I, [_VP, _I, ctypes.POINTER(TmConfig)]),
    ("tm_tune", _I, [ctypes.POINTER(_I), _I, _VP, _VP, ctypes.POINTER(TmConfig)]),
    ("tm_tune_load", _I, [ctypes.c_char_p]),
    ("tm_tune_save", _I, [ctypes.c_char_p]),
    ("tm_poll_error", _I, [_VP]),
    ("tm_selftest_wait_timeout", _I, [_LL, _VP]),
    ("tm_tc_pipeline", _I, [_I, _I] + [ctypes.POINTER(_I)] * 4),
    ("tm_tc_decode_pipeline", _I, [_I, _I] + [ctypes.POINTER(_I)] * 4),
    ("tm_decode_plan", _I, [_I, _I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_LL),
                            ctypes.POINTER(_I)]),
    ("tm_attn_decode", _I, [_VP] * 9 + [_I] * 7 + [ctypes.c_float, _I, _VP]),
    ("tm_attn_decode_plan", _I, [_I] * 6 + [ctypes.POINTER(_I)] * 2),
    ("tm_last_error", ctypes.c_char_p, []),
    ("tm_version", ctypes.c_char_p, []),
]


def lib() -> ctypes.CDLL:
    """The loaded libtmw4.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m w4a16_gemm_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _check(status: int) -> None:
    if status != TM_OK:
        raise TmError(status, lib().tm_last_error().decode())


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


_DT = {torch.float16: TM_F16, torch.bfloat16: TM_BF16}
_TORCH_DT = {TM_F16: torch.float16, TM_BF16: torch.bfloat16}


class PackedW4:
    """Library-owned packed int4 weight (freed on ``free()`` or garbage collection)."""

    def __init__(self, handle: int, K: int, N: int, group: int, dtype: torch.dtype, symmetric: bool,
                 device: torch.device):
        self.handle = handle
        self.K, self.N, self.group, self.dtype = K, N, group, dtype
        self.symmetric = symmetric
        self.device = device
        self.bits, self.fp8 = 4, False

    def info(self) -> TmPackedInfo:
        inf = TmPackedInfo()
        _check(lib().tm_packed_get(self.handle, ctypes.byref(inf)))
        return inf

    def free(self, stream=None) -> None:
        if self.handle:
            with torch.cuda.device(self.device):
                _check(lib().tm_packed_free(self.handle, _stream(stream)))
            self.handle = None

    def __del__(self):
        try:
            if self.handle and _LIB is not None:
                with torch.cuda.device(self.device):
                    _LIB.tm_packed_free(self.handle, None)
                self.handle = None
        except Exception:  # interpreter shutdown
            pass

    def raw_bytes(self) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor | None]:
        """Device copies of (qweight u8, scales u8, zeros u8 or None) for inspection."""
        inf = self.info()
        torch.cuda.synchronize(self.device)
        out = []
        for ptr, n in ((inf.qweight, inf.qweight_bytes), (inf.scales, inf.scales_bytes),
                       (inf.zeros, inf.zeros_bytes)):
            if not ptr:
                out.append(None)
                continue
            out.append(_copy_device_range(ptr, n, self.device))
        return tuple(out)


class _DevBuf:
    """Exposes a raw device range through __cuda_array_interface__ (view; never written through)."""

    def __init__(self, ptr: int, nbytes: int):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False),
                                         "version": 3, "strides": None}


def _copy_device_range(ptr: int, nbytes: int, device) -> torch.Tensor:
    """A torch copy of nbytes at device address ptr."""
    view = torch.as_tensor(_DevBuf(ptr, nbytes), device=device)
    return view.clone()


def pack(q: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor | None, group: int,
         stream=None) -> PackedW4:
    """tm_pack_w4: q [K,N] uint8, scales [K/G,N] fp16/bf16, zeros [K/G,N] uint8 or None."""
    if q.dtype != torch.uint8 or q.dim() != 2 or not q.is_cuda:
        raise ValueError("q must be a 2-D uint8 CUDA tensor")
    if scales.dtype not in _DT:
        raise ValueError("scales must be float16 or bfloat16")
    K, N = q.shape
    q = q.contiguous()
    scales = scales.contiguous()
    zp = None
    if zeros is not None:
        zeros = zeros.contiguous()
        zp = zeros.data_ptr()
    h = ctypes.c_void_p()
    with torch.cuda.device(q.device):
        _check(lib().tm_pack_w4(q.data_ptr(), scales.data_ptr(), zp, K, N, group, _DT[scales.dtype],
                                _stream(stream), ctypes.byref(h)))
    return _packed(h.value, K, N, scales.dtype, zeros is None, q.device)


def _packed(handle: int, K: int, N: int, dtype: torch.dtype, symmetric: bool, device) -> PackedW4:
    W = PackedW4(handle, K, N, 0, dtype, symmetric, device)
    inf = W.info()
    W.group = inf.group             # the group the kernels run with
    W.bits, W.fp8 = inf.bits, bool(inf.fp8)
    return W


def _codes_2d(q: torch.Tensor) -> torch.Tensor:
    if q.dtype != torch.uint8 or q.dim() != 2 or not q.is_cuda:
        raise ValueError("q must be a 2-D uint8 CUDA tensor")
    return q.contiguous()


def pack_w8(q: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor | None, group: int,
            stream=None) -> PackedW4:
    """tm_pack_w8: int8 codes q [K,N] uint8 (0..255), scales [K/G,N], zeros [K/G,N] uint8 or None."""
    q = _codes_2d(q)
    if scales.dtype not in _DT:
        raise ValueError("scales must be float16 or bfloat16")
    K, N = q.shape
    scales = scales.contiguous()
    zp = None if zeros is None else _codes_2d(zeros).data_ptr()
    h = ctypes.c_void_p()
    with torch.cuda.device(q.device):
        _check(lib().tm_pack_w8(q.data_ptr(), scales.data_ptr(), zp, K, N, group, _DT[scales.dtype],
                                _stream(stream), ctypes.byref(h)))
    return _packed(h.value, K, N, scales.dtype, zeros is None, q.device)


def pack_fp8(q: torch.Tensor, scales: torch.Tensor, group: int, stream=None) -> PackedW4:
    """tm_pack_fp8: FP8 E4M3 codes q [K,N] uint8 (bit patterns), scales [K/G,N]."""
    q = _codes_2d(q)
    if scales.dtype not in _DT:
        raise ValueError("scales must be float16 or bfloat16")
    K, N = q.shape
    scales = scales.contiguous()
    h = ctypes.c_void_p()
    with torch.cuda.device(q.device):
        _check(lib().tm_pack_fp8(q.data_ptr(), scales.data_ptr(), K, N, group, _DT[scales.dtype],
                                 _stream(stream), ctypes.byref(h)))
    return _packed(h.value, K, N, scales.dtype, True, q.device)


def _int32_2d(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.int32 or t.dim() != 2 or not t.is_cuda:
        raise ValueError(f"{name} must be a 2-D int32 CUDA tensor")
    return t.contiguous()


def pack_awq(qweight: torch.Tensor, qzeros: torch.Tensor | None, scales: torch.Tensor, group: int,
             stream=None) -> PackedW4:
    """tm_pack_awq: qweight int32 [K, N/8], qzeros int32 [K/G, N/8] or None,
    scales [K/G, N] fp16/bf16 (AWQ "GEMM" layout)."""
    qweight = _int32_2d(qweight, "qweight")
    if scales.dtype not in _DT:
        raise ValueError("scales must be float16 or bfloat16")
    K, N = qweight.shape[0], qweight.shape[1] * 8
    scales = scales.contiguous()
    zp = None if qzeros is None else _int32_2d(qzeros, "qzeros").data_ptr()
    h = ctypes.c_void_p()
    with torch.cuda.device(qweight.device):
        _check(lib().tm_pack_awq(qweight.data_ptr(), zp, scales.data_ptr(), K, N, group, _DT[scales.dtype],
                                 _stream(stream), ctypes.byref(h)))
    return _packed(h.value, K, N, scales.dtype, qzeros is None, qweight.device)


def pack_gptq(qweight: torch.Tensor, qzeros: torch.Tensor | None, scales: torch.Tensor, group: int,
              zero_offset: int = 1, stream=None) -> PackedW4:
    """tm_pack_gptq: qweight int32 [K/8, N], qzeros int32 [K/G, N/8] or None,
    scales [K/G, N] fp16/bf16; zero_offset is added to every stored zero."""
    qweight = _int32_2d(qweight, "qweight")
    if scales.dtype not in _DT:
        raise ValueError("scales must be float16 or bfloat16")
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    scales = scales.contiguous()
    zp = None if qzeros is None else _int32_2d(qzeros, "qzeros").data_ptr()
    h = ctypes.c_void_p()
    with torch.cuda.device(qweight.device):
        _check(lib().tm_pack_gptq(qweight.data_ptr(), zp, scales.data_ptr(), zero_offset, K, N, group,
                                  _DT[scales.dtype], _stream(stream), ctypes.byref(h)))
    return _packed(h.value, K, N, scales.dtype, qzeros is None, qweight.device)


def gemm(A: torch.Tensor, W: PackedW4, out: torch.Tensor | None = None, config: dict | None = None,
         stream=None) -> torch.Tensor:
    """tm_gemm_w4a16 (or _ex with an explicit variant): C = A @ dequant(W)."""
    if A.dim() != 2 or A.dtype != W.dtype or not A.is_cuda:
        raise ValueError("A must be a 2-D CUDA tensor of the weight's dtype")
    M, K = A.shape
    A = A.contiguous()
    if out is None:
        out = torch.empty((M, W.N), dtype=W.dtype, device=A.device)
    st = _stream(stream)
    if config is None:
        _check(lib().tm_gemm_w4a16(A.data_ptr(), W.handle, out.data_ptr(), M, W.N, K, st))
    else:
        c = make_config(**config)
        _check(lib().tm_gemm_w4a16_ex(A.data_ptr(), W.handle, out.data_ptr(), M, W.N, K,
                                      ctypes.byref(c), st))
    return out


def make_config(kernel="tc", block_m=16, split_k=1, dq_warps=0) -> TmConfig:
    k = {"auto": TM_KERNEL_AUTO, "gemv": TM_KERNEL_GEMV, "tc": TM_KERNEL_TC,
         "tc_decode": TM_KERNEL_TC_DECODE, "decode_mma": TM_KERNEL_DECODE_MMA}.get(kernel, kernel)
    return TmConfig(int(k), int(block_m), int(split_k), int(dq_warps))


def dequant(W: PackedW4, stream=None) -> torch.Tensor:
    """tm_dequant_w4: the full [K, N] 16-bit weight."""
    out = torch.empty((W.K, W.N), dtype=W.dtype, device=W.device)
    _check(lib().tm_dequant_w4(W.handle, out.data_ptr(), _stream(stream)))
    return out


def select(W: PackedW4, M: int) -> dict:
    """The variant tm_gemm_w4a16 runs for this weight and M."""
    c = TmConfig()
    _check(lib().tm_select(W.handle, int(M), ctypes.byref(c)))
    return c.as_dict()


def tune(W: PackedW4, Ms, stream=None) -> list[dict]:
    """tm_tune: measure every legal variant for each M; returns the chosen variants."""
    Ms = [int(m) for m in Ms]
    arr = (ctypes.c_int * len(Ms))(*Ms)
    best = (TmConfig * len(Ms))()
    _check(lib().tm_tune(arr, len(Ms), W.handle, _stream(stream), best))
    return [b.as_dict() for b in best]


def poll_error(stream=None) -> None:
    """tm_poll_error: raise TmError if a device-side condition was recorded."""
    _check(lib().tm_poll_error(_stream(stream)))


def poll_status(stream=None) -> int:
    """tm_poll_error as a plain status code."""
    return int(lib().tm_poll_error(_stream(stream)))


def selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(lib().tm_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def tc_pipeline(block_m: int, dq_warps: int) -> dict:
    """Pipeline geometry of a tcgen05 variant (no GPU needed)."""
    v = [ctypes.c_int() for _ in range(4)]
    _check(lib().tm_tc_pipeline(int(block_m), int(dq_warps), *[ctypes.byref(x) for x in v]))
    return {"stages": v[0].value, "kblocks_per_stage": v[1].value, "tmem_slots": v[2].value,
            "legal": bool(v[3].value)}


def tc_decode_pipeline(block_m: int, dq_warps: int) -> dict:
    """Pipeline geometry of a tcgen05 decode variant (no GPU needed)."""
    v = [ctypes.c_int() for _ in range(4)]
    _check(lib().tm_tc_decode_pipeline(int(block_m), int(dq_warps), *[ctypes.byref(x) for x in v]))
    return {"weight_stages": v[0].value, "act_stages_per_wg": v[1].value,
            "tmem_slots_per_wg": v[2].value, "legal": bool(v[3].value)}


def decode_plan(M: int, N: int, K: int, block_m: int, sm_count: int) -> dict:
    """Stream-K plan of the tcgen05 decode kernel (no GPU needed)."""
    g, p = ctypes.c_int(), ctypes.c_int()
    t = ctypes.c_longlong()
    _check(lib().tm_decode_plan(int(M), int(N), int(K), int(block_m), int(sm_count),
                                ctypes.byref(g), ctypes.byref(t), ctypes.byref(p)))
    return {"grid": g.value, "tiles": t.value, "partial_slots": p.value}


def attn_decode(q: torch.Tensor, k_cache: torch.Tensor, k_scale: torch.Tensor, k_zero: torch.Tensor,
                v_cache: torch.Tensor, v_scale: torch.Tensor, v_zero: torch.Tensor, lens: torch.Tensor,
                kv_bits: int, sm_scale: float, out: torch.Tensor | None = None, chunk_tiles: int = 0,
                stream=None) -> torch.Tensor:
    """tm_attn_decode: q [B, Hq, 128]; caches [B, Hkv, L_max, 128 * kv_bits / 8] uint8; scales
    [B, Hkv, L_max] of q's dtype; zeros [B, Hkv, L_max] uint8; lens [B] int32 (device)."""
    if q.dim() != 3 or q.dtype not in _DT or not q.is_cuda:
        raise ValueError("q must be a 3-D float16/bfloat16 CUDA tensor")
    B, Hq, D = q.shape
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must be 4-D and of the same shape")
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    for t in (k_cache, v_cache, k_zero, v_zero):
        if t.dtype != torch.uint8:
            raise ValueError("caches and zeros must be uint8")
    for t in (k_scale, v_scale):
        if t.dtype != q.dtype:
            raise ValueError("scales must have q's dtype")
    if lens.dtype != torch.int32:
        raise ValueError("lens must be int32")
    q = q.contiguous()
    if out is None:
        out = torch.empty_like(q)
    st = _stream(stream)
    with torch.cuda.device(q.device):
        _check(lib().tm_attn_decode(q.data_ptr(), k_cache.data_ptr(), k_scale.data_ptr(), k_zero.data_ptr(),
                                    v_cache.data_ptr(), v_scale.data_ptr(), v_zero.data_ptr(), lens.data_ptr(),
                                    out.data_ptr(), B, Hq, Hkv, D, L_max, int(kv_bits), _DT[q.dtype],
                                    float(sm_scale), int(chunk_tiles), st))
    return out


def attn_decode_plan(B: int, Hq: int, Hkv: int, L_max: int, kv_bits: int, dtype=torch.float16) -> dict:
    """tm_attn_decode_plan: the automatic chunk_tiles and the grid."""
    ct, grid = ctypes.c_int(), ctypes.c_int()
    _check(lib().tm_attn_decode_plan(B, Hq, Hkv, L_max, kv_bits, _DT[dtype], ctypes.byref(ct), ctypes.byref(grid)))
    return {"chunk_tiles": ct.value, "grid": grid.value}


def version() -> str:
    return lib().tm_version().decode()


@dataclass
class Problem:
    """Device tensors of one quantized weight (helper for tests and the bench)."""

    q: torch.Tensor
    scales: torch.Tensor
    zeros: torch.Tensor | None
    group: int
    dtype: torch.dtype


def to_device(qw, device="cuda") -> Problem:
    """Moves a synth.QuantWeight to the GPU as torch tensors."""
    dt = torch.float16 if qw.dtype == "f16" else torch.bfloat16
    q = torch.from_numpy(qw.q).to(device)
    s = torch.from_numpy(qw.scales.view("int16")).to(device).view(dt)
    z = None if qw.zeros is None else torch.from_numpy(qw.zeros).to(device)
    return Problem(q, s, z, qw.group, dt)


def acts_to_device(a_bits, dtype: torch.dtype, device="cuda") -> torch.Tensor:
    return torch.from_numpy(a_bits.view("int16")).to(device).view(dtype)

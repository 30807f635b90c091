"""The C-ABI library builds, loads without a GPU and exports every symbol
declared in include/tmw4.h; host-side argument checks answer without CUDA."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "tmw4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tm_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from w4a16_gemm_gb300 import build, binding

    build.build()
    return binding.lib()


def test_header_declares_the_documented_calls():
    names = declared_symbols()
    for n in ("tm_pack_w4", "tm_gemm_w4a16", "tm_dequant_w4", "tm_packed_free", "tm_tune",
              "tm_poll_error", "tm_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_signatures_cover_the_header():
    from w4a16_gemm_gb300 import binding

    assert sorted(n for n, _, _ in binding.SIGNATURES) == declared_symbols()


def test_host_side_validation_without_gpu(lib):
    from w4a16_gemm_gb300 import binding as b

    assert lib.tm_version().decode().startswith("tmw4")
    h = ctypes.c_void_p()
    # NULL out pointer / NULL inputs / bad group: rejected before any CUDA call
    assert lib.tm_pack_w4(None, None, None, 64, 128, 128, 0, None, None) == b.TM_ERR_INVALID_ARG
    assert lib.tm_pack_w4(None, None, None, 64, 128, 128, 0, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG
    assert lib.tm_pack_w4(16, 16, None, 256, 128, 96, 0, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG
    assert b"group" in lib.tm_last_error()
    assert lib.tm_pack_w4(16, 16, None, 256, 100, 128, 0, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG
    assert lib.tm_pack_w4(17, 16, None, 256, 128, 128, 0, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG
    assert lib.tm_gemm_w4a16(None, None, None, 1, 128, 128, None) == b.TM_ERR_INVALID_ARG
    assert lib.tm_dequant_w4(None, None, None) == b.TM_ERR_INVALID_ARG
    assert lib.tm_packed_get(None, None) == b.TM_ERR_INVALID_ARG
    assert lib.tm_select(None, 1, None) == b.TM_ERR_INVALID_ARG
    assert lib.tm_packed_free(None, None) == b.TM_OK
    # a forged handle is refused by its magic number
    fake = (ctypes.c_uint32 * 32)()
    assert lib.tm_gemm_w4a16(16, ctypes.addressof(fake), 16, 1, 128, 128, None) == b.TM_ERR_INVALID_ARG
    assert lib.tm_selftest_wait_timeout(5, None) == b.TM_ERR_INVALID_ARG


def test_attention_argument_checks_without_gpu(lib):
    """tm_attn_decode and its plan refuse bad shapes before any CUDA call."""
    from w4a16_gemm_gb300 import binding as b

    def call(B=2, Hq=8, Hkv=2, D=128, L=128, bits=8, dt=0, scale=0.1, ct=0):
        return lib.tm_attn_decode(*([None] * 9), B, Hq, Hkv, D, L, bits, dt, scale, ct, None)

    assert call(Hq=6, Hkv=4) == b.TM_ERR_INVALID_ARG             # Hq not a multiple of Hkv
    assert call(Hq=34, Hkv=2) == b.TM_ERR_UNSUPPORTED            # 17 query heads per KV head
    assert call(D=64) == b.TM_ERR_UNSUPPORTED
    assert call(bits=6) == b.TM_ERR_INVALID_ARG
    assert call(dt=7) == b.TM_ERR_INVALID_ARG
    assert call(L=100) == b.TM_ERR_INVALID_ARG                   # not a multiple of 64
    assert call(ct=-1) == b.TM_ERR_INVALID_ARG
    assert call(scale=float("nan")) == b.TM_ERR_INVALID_ARG
    assert call(B=5000) == b.TM_ERR_UNSUPPORTED                  # more sequences than the scan holds
    assert call(B=-1) == b.TM_ERR_INVALID_ARG
    assert call(B=4096, Hkv=8, Hq=8, L=65536 + 64) == b.TM_ERR_UNSUPPORTED   # rows beyond 2^31
    assert call(B=0) == b.TM_OK                                  # nothing to do
    assert call(B=1) == b.TM_ERR_INVALID_ARG                     # NULL pointers
    ct, grid = ctypes.c_int(), ctypes.c_int()
    assert lib.tm_attn_decode_plan(0, 8, 2, 128, 8, 0, ctypes.byref(ct), ctypes.byref(grid)) == b.TM_ERR_INVALID_ARG
    assert lib.tm_attn_decode_plan(2, 8, 2, 100, 8, 0, ctypes.byref(ct), ctypes.byref(grid)) == b.TM_ERR_INVALID_ARG


def test_8bit_and_checkpoint_packers_refuse_bad_arguments_without_gpu(lib):
    from w4a16_gemm_gb300 import binding as b

    h = ctypes.c_void_p()
    assert lib.tm_pack_w8(16, 16, None, 256, 128, 128, 0, None, None) == b.TM_ERR_INVALID_ARG       # NULL out
    assert lib.tm_pack_w8(None, 16, None, 256, 128, 128, 0, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG
    assert lib.tm_pack_w8(16, 16, None, 256, 128, 96, 0, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG
    assert lib.tm_pack_w8(16, 16, None, 256, 100, 128, 0, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG
    assert lib.tm_pack_fp8(16, 16, 256, 128, 128, 5, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG  # dtype
    assert lib.tm_pack_awq(None, None, 16, 256, 128, 128, 0, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG
    assert lib.tm_pack_gptq(16, None, 16, 1, 256, 128, 100, 0, None, ctypes.byref(h)) == b.TM_ERR_INVALID_ARG

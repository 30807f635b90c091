"""The GEMM entry point for callers that cannot allocate device memory.

tm_gemm_w4a16_noalloc serves applications that own all GPU memory through
their own pool (or capture a stream while the regular workspace would have
to grow): its split-K scratch is a fixed static device array of the library.
These tests call it through the C ABI and compare it with tm_gemm_w4a16 on
the same inputs, twice in a row (the scratch keeps the previous call's
contents), within the GEMM tolerance used throughout the test-suite.  The
file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests._util import TORCH_DT, c_values, packed_from
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TOL = 1e-2
STATIC_WS_BYTES = 8 << 20


def _noalloc(A, W, out):
    st = torch.cuda.current_stream().cuda_stream
    M, K = A.shape
    return binding.lib().tm_gemm_w4a16_noalloc(A.data_ptr(), W.handle, out.data_ptr(), M, W.N, K, st)


def _needed_scratch(W, M):
    """Split-K scratch bytes the selected variant uses (0 without split-K)."""
    cfg = binding.select(W, M)
    KB = W.K // 64
    gran = 1
    if cfg["kernel"] == "tc":
        gran = 4 if cfg["block_m"] <= 16 else 2 if cfg["block_m"] <= 64 else 1
    per = -(-KB // cfg["split_k"])
    per = -(-per // gran) * gran
    splits = -(-KB // per)
    return 0 if splits == 1 else splits * M * W.N * 4


@pytest.mark.parametrize("M,K,N,dt", [(4, 4096, 4096, "f16"), (16, 14336, 4096, "f16"),
                                      (1, 256, 256, "f16"), (300, 1024, 512, "bf16")])
def test_matches_the_allocating_entry_point_twice(M, K, N, dt):
    qw, a = synth.random_problem(40 + M, M, K, N, 128, dt)
    W = packed_from(qw)
    A = binding.acts_to_device(a, TORCH_DT[dt])
    ref = binding.gemm(A, W)
    torch.cuda.synchronize()
    c_ref = c_values(ref)
    assert _needed_scratch(W, M) <= STATIC_WS_BYTES
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=TORCH_DT[dt], device="cuda")
        assert _noalloc(A, W, out) == binding.TM_OK, binding.lib().tm_last_error()
        torch.cuda.synchronize()
        c = c_values(out)
        assert np.all(np.isfinite(c))
        assert oracle.max_err_ratio(c, c_ref, rel=TOL) <= 1.0
    # and against the oracle itself
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, dt)
    assert oracle.max_err_ratio(c, oracle.gemm_ref(a, w, dt), rel=TOL) <= 1.0


def test_rejects_shapes_beyond_the_static_scratch():
    M, K, N = 64, 14336, 4096
    qw, a = synth.random_problem(50, M, K, N)
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.float16)
    out = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    status = _noalloc(A, W, out)
    if _needed_scratch(W, M) > STATIC_WS_BYTES:
        assert status == binding.TM_ERR_UNSUPPORTED
        assert b"static scratch" in binding.lib().tm_last_error()
    else:
        assert status == binding.TM_OK


def test_m_zero_and_bad_arguments():
    qw, _ = synth.random_problem(51, 1, 256, 256)
    W = packed_from(qw)
    A = torch.zeros((0, 256), dtype=torch.float16, device="cuda")
    out = torch.zeros((0, 256), dtype=torch.float16, device="cuda")
    assert _noalloc(A, W, out) == binding.TM_OK
    st = torch.cuda.current_stream().cuda_stream
    assert binding.lib().tm_gemm_w4a16_noalloc(None, W.handle, None, 1, 256, 256, st) == \
        binding.TM_ERR_INVALID_ARG

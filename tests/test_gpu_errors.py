"""Device-side failure detection without faulting the GPU: the bounded wait
used by every kernel gives up, reports TM_ERR_TIMEOUT through the error word,
and the context stays usable."""

import numpy as np
import pytest
import torch

import oracle
from tests._util import TORCH_DT, gemm_poisoned, c_values, packed_from
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    assert binding.poll_status() == binding.TM_OK
    binding.selftest_wait_timeout(2_000_000)          # 2 ms, nothing ever arrives
    assert binding.poll_status() == binding.TM_ERR_TIMEOUT
    assert binding.poll_status() == binding.TM_OK     # the word was cleared
    qw, a = synth.random_problem(12, 8, 512, 256)
    W = packed_from(qw)
    C = gemm_poisoned(binding.acts_to_device(a, TORCH_DT["f16"]), W)
    torch.cuda.synchronize()
    c_ref = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16"), "f16")
    assert oracle.max_err_ratio(c_values(C), c_ref) <= 1.0


def test_selftest_limit_is_validated():
    with pytest.raises(binding.TmError):
        binding.selftest_wait_timeout(10)


def test_mismatched_shape_is_rejected():
    qw, a = synth.random_problem(13, 2, 256, 256)
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.float16)
    C = torch.empty((2, 256), dtype=torch.float16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert binding.lib().tm_gemm_w4a16(A.data_ptr(), W.handle, C.data_ptr(), 2, 384, 256, st) == \
        binding.TM_ERR_INVALID_ARG
    assert binding.lib().tm_gemm_w4a16(A.data_ptr(), W.handle, C.data_ptr(), -1, 256, 256, st) == \
        binding.TM_ERR_INVALID_ARG

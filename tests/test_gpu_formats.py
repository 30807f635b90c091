"""Weight formats beyond the u8 codes with G in {64, 128}: coarser groups
(per-channel G = K included), and checkpoints packed in int32 words (AWQ,
GPTQ) imported straight into the repack.  Each is checked bit for bit
through tm_dequant_w4 against the oracle's W = T(s * (q - z)), and through
GEMMs of several kernel families against the oracle's product; the oracle's
codes and zeros come from oracle/checkpoint.py unpacking the same int32
arrays the library imports."""

import numpy as np
import pytest
import torch

import oracle
from oracle import checkpoint as ck
from tests._util import (TORCH_DT, awq_pack, bits_of, c_values, gemm_poisoned, gptq_pack_qweight,
                         gptq_pack_qzeros)
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _variants(M):
    if M <= 8:
        return [None, dict(kernel="gemv", split_k=2), dict(kernel="decode_mma", split_k=0),
                dict(kernel="decode_mma", split_k=4, dq_warps=1), dict(kernel="gemv", split_k=2, dq_warps=1)]
    if M <= 16:
        return [None, dict(kernel="tc_decode", block_m=16, dq_warps=8), dict(kernel="decode_mma", split_k=1)]
    return [None, dict(kernel="tc", block_m=128, split_k=2, dq_warps=8)]


def _check_gemms(W, q, s_bits, z, G, dt, seed):
    K, N = q.shape
    w = oracle.dequant_bits(q, s_bits, z, G, dt)
    assert np.array_equal(bits_of(binding.dequant(W)), w)
    for M in (1, 16, 200):
        a = synth.random_problem(seed + M, M, K, N, 64, dt)[1]
        A = binding.acts_to_device(a, TORCH_DT[dt])
        c_ref = oracle.gemm_ref(a, w, dt)
        for cfg in _variants(M):
            C = gemm_poisoned(A, W, config=cfg)
            torch.cuda.synchronize()
            assert oracle.max_err_ratio(c_values(C), c_ref, rel=TOL) <= 1.0, (M, cfg)
    binding.poll_error()


@pytest.mark.parametrize("G,packed_G", [(768, 128), (256, 128), (192, 64), (384, 128)])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_coarse_groups(G, packed_G, dt):
    """Any multiple of 64 (per-channel: G = K = 768) is stored at the packed
    group with its scale and zero repeated: the weight is unchanged."""
    K, N = 768, 256
    qw, _ = synth.random_problem(3 + G, 1, K, N, G, dt)
    p = binding.to_device(qw)
    W = binding.pack(p.q, p.scales, p.zeros, G)
    assert W.group == packed_G and W.info().group == packed_G
    _check_gemms(W, qw.q, qw.scales, qw.zeros, G, dt, seed=11)


@pytest.mark.parametrize("G,symmetric", [(128, False), (64, False), (256, True)])
def test_awq_import(G, symmetric):
    K, N, dt = 512, 384, "f16"
    rng = np.random.default_rng(G)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = None if symmetric else rng.integers(0, 16, size=(K // G, N), dtype=np.uint8)
    s = synth.random_problem(5, 1, K, N, G, dt)[0].scales
    qweight = awq_pack(q)
    qzeros = None if z is None else awq_pack(z)
    # the oracle's codes and zeros from the int32 arrays themselves
    q_o = ck.unpack_awq(qweight)
    z_o = None if qzeros is None else ck.unpack_awq(qzeros)
    W = binding.pack_awq(torch.from_numpy(qweight).cuda(),
                         None if qzeros is None else torch.from_numpy(qzeros).cuda(),
                         torch.from_numpy(s.view(np.int16)).cuda().view(torch.float16), G)
    assert W.symmetric == symmetric
    _check_gemms(W, q_o, s, z_o, G, dt, seed=21)


@pytest.mark.parametrize("G,offset,dt", [(128, 1, "f16"), (64, 0, "bf16"), (512, 1, "f16")])
def test_gptq_import(G, offset, dt):
    K, N = 512, 256
    rng = np.random.default_rng(G + offset)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = rng.integers(offset, 16, size=(K // G, N), dtype=np.uint8)
    s = synth.random_problem(6, 1, K, N, G, dt)[0].scales
    qweight, qzeros = gptq_pack_qweight(q), gptq_pack_qzeros(z, offset)
    q_o, z_o = ck.unpack_gptq_qweight(qweight), ck.unpack_gptq_qzeros(qzeros, offset)
    W = binding.pack_gptq(torch.from_numpy(qweight).cuda(), torch.from_numpy(qzeros).cuda(),
                          torch.from_numpy(s.view(np.int16)).cuda().view(TORCH_DT[dt]), G, zero_offset=offset)
    _check_gemms(W, q_o, s, z_o, G, dt, seed=31)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_group_32(dt):
    """Groups of 32: two scales per 64-K block.  The TC kernel (any M) and the
    CUDA-core GEMV (M <= 8) run them; the kernels that scale fp32 sums per
    block refuse them."""
    K, N = 512, 256
    qw, _ = synth.random_problem(8, 1, K, N, 32, dt)
    W = packed_from_qw(qw)
    assert W.group == 32
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 32, dt)
    assert np.array_equal(bits_of(binding.dequant(W)), w)
    for M in (1, 5, 16, 200):
        a = synth.random_problem(40 + M, M, K, N, 32, dt)[1]
        A = binding.acts_to_device(a, TORCH_DT[dt])
        c_ref = oracle.gemm_ref(a, w, dt)
        cfgs = [None, dict(kernel="tc", block_m=16, split_k=2), dict(kernel="tc", block_m=128, split_k=1)]
        if M <= 8:
            cfgs += [dict(kernel="gemv", split_k=1), dict(kernel="gemv", split_k=4)]
        for cfg in cfgs:
            C = gemm_poisoned(A, W, config=cfg)
            torch.cuda.synchronize()
            assert oracle.max_err_ratio(c_values(C), c_ref, rel=TOL) <= 1.0, (M, cfg)
        if M <= 16:
            for cfg in (dict(kernel="decode_mma"), dict(kernel="tc_decode", block_m=16),
                        dict(kernel="gemv", dq_warps=1)):
                with pytest.raises(binding.TmError) as e:
                    binding.gemm(A, W, config=cfg)
                assert e.value.status == binding.TM_ERR_UNSUPPORTED, cfg
    binding.poll_error()


def packed_from_qw(qw):
    p = binding.to_device(qw)
    return binding.pack(p.q, p.scales, p.zeros, qw.group)


def test_format_errors():
    K, N = 256, 128
    q = torch.zeros((K, N), dtype=torch.uint8, device="cuda")
    s = torch.ones((K // 16, N), dtype=torch.float16, device="cuda")
    with pytest.raises(binding.TmError) as e:
        binding.pack(q, s, None, 16)                  # groups finer than 32 are not supported
    assert e.value.status == binding.TM_ERR_INVALID_ARG
    qw = torch.zeros((K // 8, N), dtype=torch.int32, device="cuda")
    s2 = torch.ones((K // 128, N), dtype=torch.float16, device="cuda")
    with pytest.raises(binding.TmError) as e:
        binding.pack_gptq(qw, None, s2, 128, zero_offset=2)
    assert e.value.status == binding.TM_ERR_INVALID_ARG
    # a stored zero of 15 plus the offset 1 is not a code: reported on the device
    qz = torch.full((K // 128, N // 8), -1, dtype=torch.int32, device="cuda")    # every nibble 15
    W = binding.pack_gptq(qw, qz, s2, 128, zero_offset=1)
    torch.cuda.synchronize()
    assert binding.poll_status() == binding.TM_ERR_INVALID_ARG
    W.free()

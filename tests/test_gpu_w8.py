"""8-bit weights (int8 with a zero point, FP8 E4M3) on the same pipeline:
packing bit for bit against oracle/w8.py, the dequant-only kernel bit for
bit, one-hot rows exactly, and GEMMs of the kernels that take them (the
CUDA-core GEMV and the tcgen05 kernel) against the oracle's product."""

import numpy as np
import pytest
import torch

import oracle
from oracle import w8
from tests._util import TORCH_DT, bits_of, c_values, gemm_poisoned
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TOL = 1e-2
NAN_CODES = (0x7F, 0xFF)


def _scales(rng, rows, N, dt, lo=2e-4, hi=2e-3):
    s = rng.uniform(lo, hi, size=(rows, N)) * rng.choice([-1.0, 1.0], size=(rows, N))
    return oracle.rne_f16_bits(s) if dt == "f16" else oracle.rne_bf16_bits(s.astype(np.float32))


def _problem(seed, K, N, G, dt, fmt):
    """(q, scales, zeros or None) with fmt 'int8', 'int8sym' or 'fp8'."""
    rng = np.random.default_rng(seed)
    if fmt == "fp8":
        q = rng.integers(0, 256, size=(K, N), dtype=np.uint8)
        q[np.isin(q, NAN_CODES)] = 0x38                      # no NaN weights
        return q, _scales(rng, K // G, N, dt, 1e-4, 1e-3), None
    q = rng.integers(0, 256, size=(K, N), dtype=np.uint8)
    z = None if fmt == "int8sym" else rng.integers(0, 256, size=(K // G, N), dtype=np.uint8)
    return q, _scales(rng, K // G, N, dt), z


def _pack(q, s, z, G, dt, fmt):
    qd = torch.from_numpy(q).cuda()
    sd = torch.from_numpy(s.view(np.int16)).cuda().view(TORCH_DT[dt])
    if fmt == "fp8":
        return binding.pack_fp8(qd, sd, G)
    return binding.pack_w8(qd, sd, None if z is None else torch.from_numpy(z).cuda(), G)


def _w_ref(q, s, z, G, dt, fmt):
    return w8.dequant8_bits(q, s, z, G, dt, fp8=(fmt == "fp8"))


@pytest.mark.parametrize("fmt", ["int8", "int8sym", "fp8"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_pack_and_dequant_bit_exact(fmt, dt):
    K, N, G = 384, 256, 128
    q, s, z = _problem(1, K, N, G, dt, fmt)
    W = _pack(q, s, z, G, dt, fmt)
    assert W.bits == 8 and W.fp8 == (fmt == "fp8") and W.symmetric == (z is None)
    qb, sb, zb = W.raw_bytes()
    assert np.array_equal(qb.cpu().numpy(), w8.pack8_ref(q))
    assert np.array_equal(sb.cpu().numpy().view(np.uint16), oracle.pack_scales_ref(s))
    if z is not None:
        assert np.array_equal(zb.cpu().numpy(), w8.pack_zeros8_ref(z))
    assert np.array_equal(bits_of(binding.dequant(W)), _w_ref(q, s, z, G, dt, fmt))
    assert binding.poll_status() == binding.TM_OK


@pytest.mark.parametrize("G", [32, 64, 256])
def test_dequant_other_groups(G):
    K, N, dt = 512, 128, "f16"
    q, s, z = _problem(2 + G, K, N, G, dt, "int8")
    W = _pack(q, s, z, G, dt, "int8")
    assert np.array_equal(bits_of(binding.dequant(W)), _w_ref(q, s, z, G, dt, "int8"))


def _variants(M, G=128):
    out = [None]
    if M <= 8:
        out += [dict(kernel="gemv", split_k=1), dict(kernel="gemv", split_k=3)]
    if M <= 16 and G >= 64:
        # register-MMA decode kernel: stream-K with one or two K-groups, clusters of 2 and 5
        out += [dict(kernel="decode_mma", split_k=0, dq_warps=4), dict(kernel="decode_mma", split_k=1, dq_warps=8),
                dict(kernel="decode_mma", split_k=2, dq_warps=1), dict(kernel="decode_mma", split_k=5, dq_warps=2)]
    out += [dict(kernel="tc", block_m=16, split_k=2, dq_warps=4), dict(kernel="tc", block_m=64, split_k=1, dq_warps=8)]
    if M > 16:
        out += [dict(kernel="tc", block_m=128, split_k=1, dq_warps=16), dict(kernel="tc", block_m=256, split_k=1, dq_warps=8)]
    return out


@pytest.mark.parametrize("fmt,dt,G", [("int8", "f16", 128), ("int8sym", "bf16", 64), ("fp8", "f16", 128),
                                      ("fp8", "bf16", 32), ("int8", "bf16", 32), ("int8", "bf16", 128),
                                      ("fp8", "bf16", 64), ("int8sym", "f16", 128)])
def test_gemm_against_the_oracle(fmt, dt, G):
    K, N = 1024, 384
    q, s, z = _problem(3, K, N, G, dt, fmt)
    W = _pack(q, s, z, G, dt, fmt)
    w = _w_ref(q, s, z, G, dt, fmt)
    for M in (1, 5, 16, 200):
        a = synth.random_problem(20 + M, M, K, N, 128, dt)[1]
        A = binding.acts_to_device(a, TORCH_DT[dt])
        c_ref = oracle.gemm_ref(a, w, dt)
        for cfg in _variants(M, G):
            C = gemm_poisoned(A, W, config=cfg)
            torch.cuda.synchronize()
            assert oracle.max_err_ratio(c_values(C), c_ref, rel=TOL) <= 1.0, (M, cfg)
    binding.poll_error()


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_one_hot_rows_reproduce_the_weight(fmt):
    K, N, G, dt = 512, 256, 128, "f16"
    q, s, z = _problem(4, K, N, G, dt, fmt)
    W = _pack(q, s, z, G, dt, fmt)
    w = _w_ref(q, s, z, G, dt, fmt)
    ks = [0, 1, 15, 16, 63, 64, 255, 511]
    a = np.zeros((len(ks), K), np.uint16)
    for i, k in enumerate(ks):
        a[i, k] = 0x3C00
    A = binding.acts_to_device(a, torch.float16)
    for cfg in [dict(kernel="gemv", split_k=1), dict(kernel="gemv", split_k=4),
                dict(kernel="tc", block_m=16, split_k=1, dq_warps=4), dict(kernel="tc", block_m=128, split_k=3),
                dict(kernel="decode_mma", split_k=0, dq_warps=4), dict(kernel="decode_mma", split_k=3, dq_warps=1)]:
        C = gemm_poisoned(A, W, config=cfg)
        torch.cuda.synchronize()
        # exact as numbers: a code equal to its zero point gives -0 for a
        # negative scale, and an fp32 sum that starts from +0 returns +0
        assert np.array_equal(c_values(C), oracle.act_bits_to_f64(w[ks], dt)), cfg
    binding.poll_error()


def test_kernels_without_8bit_refuse_and_selection_runs():
    """tc_decode and the tensor-core GEMV take 4-bit codes only, and the
    register-MMA decode kernel at most two K-groups with 8-bit codes."""
    K, N, G, dt = 512, 256, 128, "f16"
    q, s, z = _problem(5, K, N, G, dt, "int8")
    W = _pack(q, s, z, G, dt, "int8")
    A = binding.acts_to_device(np.zeros((4, K), np.uint16), torch.float16)
    for cfg in (dict(kernel="decode_mma", dq_warps=16), dict(kernel="tc_decode", block_m=16),
                dict(kernel="gemv", dq_warps=1)):
        with pytest.raises(binding.TmError) as e:
            binding.gemm(A, W, config=cfg)
        assert e.value.status == binding.TM_ERR_UNSUPPORTED, cfg
    for M in (1, 8, 16, 100):
        assert binding.select(W, M)["kernel"] in ("gemv", "decode_mma", "tc"), M
    assert binding.select(W, 16)["kernel"] == "decode_mma"
    best = binding.tune(W, [2, 12, 40])
    assert all(b["kernel"] in ("gemv", "decode_mma", "tc") for b in best)
    w = _w_ref(q, s, z, G, dt, "int8")
    for M in (2, 12, 40):
        a = synth.random_problem(60 + M, M, K, N)[1]
        C = gemm_poisoned(binding.acts_to_device(a, torch.float16), W)
        torch.cuda.synchronize()
        assert oracle.max_err_ratio(c_values(C), oracle.gemm_ref(a, w, dt), rel=TOL) <= 1.0, M

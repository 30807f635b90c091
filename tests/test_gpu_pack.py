"""GPU parity of the offline repack and the dequant-only kernel (bit-exact).

Packing follows the pages' offline weight packing (TurboMind paper,
pith.science review, Figures 6/7); the oracle's reader/writer of the packed
layout is written from the layout specification.  Dequant must equal the
oracle's W = RNE_T(s*(q-z)) bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
from tests._util import bits_of, packed_from
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

CASES = [
    # K, N, group, dtype, symmetric
    (256, 256, 128, "f16", False),
    (512, 384, 128, "bf16", False),
    (192, 128, 64, "f16", True),
    (1024, 640, 64, "bf16", True),
    (4096, 1024, 128, "f16", False),
]


@pytest.mark.parametrize("K,N,G,dt,sym", CASES)
def test_pack_and_dequant_bit_exact(K, N, G, dt, sym):
    qw, _ = synth.random_problem(K + N, 1, K, N, G, dt, sym)
    W = packed_from(qw)
    qb, sb, zb = W.raw_bytes()
    assert np.array_equal(qb.cpu().numpy(), oracle.pack_ref(qw.q))
    assert np.array_equal(sb.cpu().numpy().view(np.uint16), oracle.pack_scales_ref(qw.scales))
    if sym:
        assert zb is None
    else:
        assert np.array_equal(zb.cpu().numpy(), oracle.pack_zeros_ref(qw.zeros))
    assert np.array_equal(oracle.unpack_ref(qb.cpu().numpy(), K, N), qw.q)
    Wd = binding.dequant(W)
    torch.cuda.synchronize()
    binding.poll_error()
    want = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, G, dt)
    assert np.array_equal(bits_of(Wd), want)


def test_every_code_and_zero_with_extreme_scales():
    """All 16x16 (q, z) pairs against subnormal, power-of-two and random scales."""
    K, N, G = 256, 128, 64   # 4 groups
    rng = np.random.default_rng(77)
    for dt in ("f16", "bf16"):
        q = np.zeros((K, N), np.uint8)
        z = np.zeros((K // G, N), np.uint8)
        for n in range(N):
            z[:, n] = (n // 8 + np.arange(K // G)) % 16
            q[:, n] = (np.arange(K) + n) % 16
        if dt == "f16":
            s = rng.integers(0, 0x7C00, size=(K // G, N), dtype=np.uint16)
            s[0, :8] = [0x0001, 0x0002, 0x0200, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x1000]
        else:
            s = rng.integers(0, 0x7F00, size=(K // G, N), dtype=np.uint16)
            s[0, :6] = [0x0001, 0x007F, 0x0080, 0x3F80, 0x7F7F, 0x3B80]
        qw = synth.QuantWeight(q, s, z, G, dt)
        W = packed_from(qw)
        Wd = binding.dequant(W)
        torch.cuda.synchronize()
        with np.errstate(over="ignore"):
            want = oracle.dequant_bits(q, s, z, G, dt)
        assert np.array_equal(bits_of(Wd), want), dt


def test_full_size_pack_matches_oracle():
    qw = synth.weight("decode_8b", 2)          # K=4096, N=28672
    W = packed_from(qw)
    qb, _, zb = W.raw_bytes()
    assert np.array_equal(qb.cpu().numpy(), oracle.pack_ref(qw.q))
    assert np.array_equal(zb.cpu().numpy(), oracle.pack_zeros_ref(qw.zeros))


def test_code_above_15_is_reported():
    qw, _ = synth.random_problem(5, 1, 128, 128)
    q = qw.q.copy()
    q[3, 7] = 0x1F
    p = binding.to_device(synth.QuantWeight(q, qw.scales, qw.zeros, 128, "f16"))
    W = binding.pack(p.q, p.scales, p.zeros, 128)
    assert binding.poll_status() == binding.TM_ERR_INVALID_ARG
    qb, _, _ = W.raw_bytes()
    q_masked = q & 0xF
    assert np.array_equal(qb.cpu().numpy(), oracle.pack_ref(q_masked))
    assert binding.poll_status() == binding.TM_OK


def test_pack_argument_errors():
    q = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((2, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(binding.TmError) as e:
        binding.pack(q, s, None, 96)
    assert e.value.status == binding.TM_ERR_INVALID_ARG
    with pytest.raises(binding.TmError):
        binding.pack(q[:, :192].contiguous(), s[:, :192].contiguous(), None, 128)
    qa = torch.zeros(256 * 256 + 1, dtype=torch.uint8, device="cuda")[1:].view(256, 256)
    with pytest.raises(binding.TmError):
        binding.pack(qa, s, None, 128)

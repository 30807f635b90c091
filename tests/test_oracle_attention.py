"""Pins of the decode-attention oracle (oracle/attention.py).

Each pin checks the oracle against something other than itself: a pure-Python
brute force with rational dequantization, closed forms (one token, two
tokens with a chosen score gap, equal keys, zero softmax scale), the
grouped-query head mapping, the nibble order of 4-bit rows, and masking.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import attention as at
from tests.test_oracle_casts import round_exact
from w4a16_gemm_gb300 import synth


def _f16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def _val(bits, fmt):
    bits = int(bits)
    if fmt == "f16":
        return float(np.uint16(bits).view(np.float16))
    return float(np.uint32(bits << 16).view(np.float32))


def _brute(p: synth.KVProblem):
    """Pure-Python loops: rational dequant rounded exactly, math.exp/fsum."""
    B, Hq, D, Hkv = p.B, p.Hq, p.D, p.Hkv
    grp = Hq // Hkv
    sc = float(np.float32(p.sm_scale))
    out = np.zeros((B, Hq, D))

    def code(c, b, h, t, d):
        if p.bits == 8:
            return int(c[b, h, t, d])
        byte = int(c[b, h, t, d // 2])
        return (byte >> 4) if d % 2 else (byte & 15)

    def deq(c, s, z, b, h, t, d):
        return round_exact(Fraction(_val(s[b, h, t], p.dtype)) * (code(c, b, h, t, d) - int(z[b, h, t])), p.dtype)

    for b in range(B):
        n = int(p.lens[b])
        for hq in range(Hq):
            h = hq // grp
            if n == 0:
                continue
            qv = [_val(p.q[b, hq, d], p.dtype) for d in range(D)]
            s = []
            for t in range(n):
                k = [deq(p.k_codes, p.k_scale, p.k_zero, b, h, t, d) for d in range(D)]
                s.append(sc * math.fsum(qv[d] * k[d] for d in range(D)))
            m = max(s)
            w = [math.exp(x - m) for x in s]
            tot = math.fsum(w)
            for d in range(D):
                out[b, hq, d] = math.fsum(w[t] * deq(p.v_codes, p.v_scale, p.v_zero, b, h, t, d)
                                          for t in range(n)) / tot
    return out


def _ref(p):
    return at.attn_decode_ref(p.q, p.k_codes, p.k_scale, p.k_zero, p.v_codes, p.v_scale, p.v_zero,
                              p.lens, p.bits, p.dtype, p.sm_scale)


@pytest.mark.parametrize("bits,dtype", [(8, "f16"), (4, "f16"), (8, "bf16"), (4, "bf16")])
def test_against_brute_force(bits, dtype):
    p = synth.kv_problem(1, B=3, Hq=4, Hkv=2, D=8, lens=[5, 1, 0], L_max=64, bits=bits, dtype=dtype)
    got, want = _ref(p), _brute(p)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    assert np.all(got[2] == 0.0)          # length 0: no tokens, output 0


def test_one_token_gives_its_value_row():
    p = synth.kv_problem(2, B=2, Hq=8, Hkv=2, D=16, lens=[1, 1], L_max=64)
    got = _ref(p)
    for b in range(2):
        for hq in range(8):
            h = hq // 4
            v = at.kv_dequant_bits(p.v_codes[b, h, :1], p.v_scale[b, h, :1], p.v_zero[b, h, :1], "f16")
            assert np.array_equal(got[b, hq], v[0].view(np.float16).astype(np.float64))


def test_two_tokens_closed_form():
    """K0 = 0, K1 = s * e0 (q - z = 1 in dimension 0), Q = x * e0: the score
    gap is a = sm_scale * x * s and P = (1, e^a) / (1 + e^a)."""
    D = 8
    p = synth.kv_problem(3, B=1, Hq=1, Hkv=1, D=D, lens=[2], L_max=64)
    p.k_zero[:] = 7
    p.k_codes[:] = 7
    p.k_codes[0, 0, 1, 0] = 8
    p.k_scale[:] = _f16(0.5)
    p.q[:] = _f16(0.0)
    p.q[0, 0, 0] = _f16(1.5)
    p.sm_scale = 0.75
    a = 0.75 * 1.5 * 0.5
    w1 = math.exp(a) / (1.0 + math.exp(a))
    V = [at.kv_dequant_bits(p.v_codes[0, 0, t], p.v_scale[0, 0, t:t + 1], p.v_zero[0, 0, t:t + 1], "f16")
         .view(np.float16).astype(np.float64) for t in range(2)]
    want = (1.0 - w1) * V[0] + w1 * V[1]
    assert np.allclose(_ref(p)[0, 0], want, rtol=1e-13, atol=1e-15)


def test_equal_keys_average_the_values():
    p = synth.kv_problem(4, B=1, Hq=2, Hkv=1, D=16, lens=[37], L_max=64)
    p.k_codes[0, 0] = p.k_codes[0, 0, 0]
    p.k_scale[0, 0] = p.k_scale[0, 0, 0]
    p.k_zero[0, 0] = p.k_zero[0, 0, 0]
    V = at.kv_dequant_bits(p.v_codes[0, 0, :37], p.v_scale[0, 0, :37], p.v_zero[0, 0, :37], "f16")
    mean = V.view(np.float16).astype(np.float64).mean(axis=0)
    for hq in range(2):
        assert np.allclose(_ref(p)[0, hq], mean, rtol=1e-13, atol=1e-15)


def test_zero_softmax_scale_is_uniform():
    p = synth.kv_problem(5, B=1, Hq=1, Hkv=1, D=8, lens=[10], L_max=64)
    p.sm_scale = 0.0
    V = at.kv_dequant_bits(p.v_codes[0, 0, :10], p.v_scale[0, 0, :10], p.v_zero[0, 0, :10], "f16")
    assert np.allclose(_ref(p)[0, 0], V.view(np.float16).astype(np.float64).mean(axis=0), rtol=1e-13)


def test_grouped_query_head_mapping():
    """Hq = 8 over Hkv = 2: V of KV head h is the constant h + 1, so query
    head hq must read exactly hq // 4 + 1."""
    p = synth.kv_problem(6, B=1, Hq=8, Hkv=2, D=8, lens=[9], L_max=64)
    p.v_codes[:] = 0
    p.v_zero[:] = 0
    p.v_codes[0, 0] = 1
    p.v_codes[0, 1] = 2
    p.v_scale[:] = _f16(1.0)
    got = _ref(p)
    for hq in range(8):
        assert np.allclose(got[0, hq], hq // 4 + 1, rtol=1e-14, atol=0), hq


def test_kv4_nibble_order():
    assert at.unpack_kv4(np.array([0x21, 0xF0], np.uint8)).tolist() == [1, 2, 0, 15]
    c = np.random.default_rng(0).integers(0, 16, size=(3, 10), dtype=np.uint8)
    assert np.array_equal(at.unpack_kv4(at.pack_kv4(c)), c)
    # a 4-bit row reads the same as its unpacked 8-bit twin
    p4 = synth.kv_problem(7, B=1, Hq=2, Hkv=1, D=16, lens=[6], L_max=64, bits=4)
    p8 = synth.kv_problem(7, B=1, Hq=2, Hkv=1, D=16, lens=[6], L_max=64, bits=8)
    for a in ("q", "k_scale", "k_zero", "v_scale", "v_zero"):
        setattr(p8, a, getattr(p4, a))
    p8.k_codes = at.unpack_kv4(p4.k_codes)
    p8.v_codes = at.unpack_kv4(p4.v_codes)
    assert np.array_equal(_ref(p4), _ref(p8))


def test_tokens_past_the_length_are_ignored():
    p = synth.kv_problem(8, B=2, Hq=4, Hkv=1, D=16, lens=[11, 64], L_max=64)
    base = _ref(p)
    p.k_codes[0, :, 11:] = 255
    p.v_codes[0, :, 11:] = 255
    p.k_scale[0, :, 11:] = _f16(np.inf)
    p.v_scale[0, :, 11:] = _f16(np.nan)
    assert np.array_equal(_ref(p), base)


def test_kv_dequant_matches_rational_rounding():
    rng = np.random.default_rng(9)
    for fmt in ("f16", "bf16"):
        codes = rng.integers(0, 256, size=(50, 4), dtype=np.uint8)
        z = rng.integers(0, 256, size=50, dtype=np.uint8)
        sbits = synth.to_16bit(rng.uniform(-3, 3, size=50).astype(np.float32), fmt)
        got = at.kv_dequant_bits(codes, sbits, z, fmt)
        for t in range(50):
            for d in range(4):
                want = round_exact(Fraction(_val(sbits[t], fmt)) * (int(codes[t, d]) - int(z[t])), fmt)
                assert _val(got[t, d], fmt) == want

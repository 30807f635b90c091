"""Pins of the 8-bit weight oracle (oracle/w8.py)."""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import w8
from tests.test_oracle_casts import round_exact


def test_e4m3_against_torch_and_by_hand():
    codes = np.arange(256, dtype=np.uint8)
    ours = w8.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.isnan(ours[[0x7F, 0xFF]]).all() and np.isnan(ours).sum() == 2
    assert ours[0x38] == 1.0 and ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9
    assert ours[0x08] == 2.0 ** -6 and ours[0xB8] == -1.0
    assert ours[0x80] == 0.0 and np.signbit(ours[0x80])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_int8_unit_steps_reproduce_the_scale(dtype):
    """q - z = +1 gives exactly s, -1 gives -s, 0 gives +0, for every z."""
    rng = np.random.default_rng(3)
    N = 128
    s_bits = (rng.integers(0x2000, 0x5800, size=(1, N)) if dtype == "f16"
              else rng.integers(0x3800, 0x4400, size=(1, N))).astype(np.uint16)
    for d, want in ((1, s_bits), (-1, s_bits ^ np.uint16(0x8000)), (0, np.zeros_like(s_bits))):
        for z0 in (0, 1, 127, 128, 200, 254):
            if not 0 <= z0 + d <= 255:
                continue
            q = np.full((64, N), z0 + d, dtype=np.uint8)
            z = np.full((1, N), z0, dtype=np.uint8)
            w = w8.dequant8_bits(q, s_bits, z, 64, dtype)
            assert np.array_equal(w, np.repeat(want, 64, axis=0)), (d, z0)
    # symmetric: the zero point is 128
    q = np.full((64, N), 129, dtype=np.uint8)
    assert np.array_equal(w8.dequant8_bits(q, s_bits, None, 64, dtype), np.repeat(s_bits, 64, axis=0))


def test_fp8_with_unit_scale_is_the_code_value():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    q = np.tile(codes[:, None], (1, 128))[:64 * (len(codes) // 64)]
    s = np.full((q.shape[0] // 64, 128), 0x3C00, dtype=np.uint16)      # fp16 1.0
    w = w8.dequant8_bits(q, s, None, 64, "f16", fp8=True)
    ref = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).to(torch.float16).numpy().view(np.uint16)
    assert np.array_equal(w, ref)
    with pytest.raises(ValueError):
        w8.dequant8_f64(q, s, np.zeros_like(s, dtype=np.uint8), 64, "f16", fp8=True)


def test_pack8_layout_properties():
    rng = np.random.default_rng(4)
    K, N = 192, 256
    q = rng.integers(0, 256, size=(K, N), dtype=np.uint8)
    p = w8.pack8_ref(q)
    assert p.size == K * N
    assert np.array_equal(w8.unpack8_ref(p, K, N), q)
    # block (nt, kb) is 8192 contiguous bytes; chunk kq*128 + c is 16 consecutive K of column c
    KB = K // 64
    for nt, kb, kq, c in ((0, 0, 0, 0), (1, 2, 3, 127), (0, 1, 2, 5), (1, 0, 1, 64)):
        off = (nt * KB + kb) * 8192 + (kq * 128 + c) * 16
        assert np.array_equal(p[off:off + 16], q[64 * kb + 16 * kq: 64 * kb + 16 * kq + 16, 128 * nt + c])
    # one-hot: a single nonzero byte lands at exactly one place
    q1 = np.zeros((K, N), dtype=np.uint8)
    q1[70, 130] = 9
    p1 = w8.pack8_ref(q1)
    assert np.count_nonzero(p1) == 1
    assert p1[(1 * KB + 1) * 8192 + (0 * 128 + 2) * 16 + 6] == 9


def test_pack_zeros8():
    z = np.arange(3 * 256, dtype=np.uint32).reshape(3, 256).astype(np.uint8)
    zp = w8.pack_zeros8_ref(z)
    assert zp[(1 * 3 + 2) * 128 + 5] == z[2, 128 + 5]


def _e4m3_by_hand(c: int):
    """E4M3 from its bit layout: 1 sign, 4 exponent (bias 7), 3 mantissa bits;
    exponent 0 is subnormal; S.1111.111 is NaN; no infinities."""
    sign = -1 if c & 0x80 else 1
    e, m = (c >> 3) & 0xF, c & 0x7
    if e == 0xF and m == 0x7:
        return None
    if e == 0:
        return sign * Fraction(m, 8) * Fraction(1, 2 ** 6)
    return sign * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def _scales(fmt, n, seed):
    rng = np.random.default_rng(seed)
    hi = 0x7C00 if fmt == "f16" else 0x7F80
    bits = rng.integers(0, hi, size=n).astype(np.uint16)
    sign = rng.integers(0, 2, size=n).astype(np.uint16) << 15
    return bits | sign


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_int8_every_difference_vs_rational(fmt):
    """Every q - z in [-255, 255] (each from a random valid (q, z)) times a
    spread of scales, subnormal to large, either sign, against the exactly
    rounded rational product."""
    rng = np.random.default_rng(21)
    d = np.arange(-255, 256)
    z = np.array([rng.integers(max(0, -x), min(255, 255 - x) + 1) for x in d], dtype=np.int64)
    q = (z + d).astype(np.uint8)
    z = z.astype(np.uint8)
    scales = _scales(fmt, 40, 22 if fmt == "f16" else 23)
    S = scales.size
    Q = np.repeat(q[:, None], S, axis=1)
    Z = np.repeat(z[:, None], S, axis=1)              # group = 1: one zero per row
    Sc = np.repeat(scales[None, :], d.size, axis=0)
    with np.errstate(over="ignore"):
        got = oracle.act_bits_to_f64(w8.dequant8_bits(Q, Sc, Z, 1, fmt), fmt)
    sval = oracle.act_bits_to_f64(scales, fmt)
    for i, dd in enumerate(d):
        want = [round_exact(Fraction(float(sv)) * int(dd), fmt) for sv in sval]
        assert np.array_equal(got[i], np.array(want)), dd


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_fp8_every_code_vs_rational(fmt):
    codes = np.array([c for c in range(256) if _e4m3_by_hand(c) is not None], dtype=np.uint8)
    assert codes.size == 254
    hand = w8.e4m3_to_f64(codes)
    assert [Fraction(float(x)) for x in hand] == [_e4m3_by_hand(int(c)) for c in codes]
    scales = _scales(fmt, 24, 24 if fmt == "f16" else 25)
    S = scales.size
    Q = np.repeat(codes[:, None], S, axis=1)
    Sc = np.repeat(scales[None, :], codes.size, axis=0)
    with np.errstate(over="ignore"):
        got = oracle.act_bits_to_f64(w8.dequant8_bits(Q, Sc, None, 1, fmt, fp8=True), fmt)
    sval = oracle.act_bits_to_f64(scales, fmt)
    for i, c in enumerate(codes):
        v = _e4m3_by_hand(int(c))
        want = [round_exact(Fraction(float(sv)) * v, fmt) for sv in sval]
        assert np.array_equal(got[i], np.array(want)), hex(c)

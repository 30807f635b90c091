"""Pins for the oracle's dequantization W = RNE_T(s * (q - z)).

Follows the runtime "I2F conversion and scaling" of packed int4 values
(TurboMind paper, pith.science review, Figure 6; Figure 4 text).  Pinned by an
exhaustive closed-form check against exact rational arithmetic, and by the
special cases q == z (exact zero) and symmetric == asymmetric with z = 8.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.test_oracle_casts import round_exact


def _scale_set(fmt, n, seed):
    rng = np.random.default_rng(seed)
    if fmt == "f16":
        # all exponents incl. subnormal scales, plus powers of two
        bits = rng.integers(0, 0x7C00, size=n, dtype=np.uint16)
        pow2 = np.array([0x0001, 0x0200, 0x0400, 0x1000, 0x3C00, 0x5000], dtype=np.uint16)
    else:
        bits = rng.integers(0, 0x7F80, size=n, dtype=np.uint16)
        pow2 = np.array([0x0001, 0x0080, 0x3F80, 0x3B80, 0x4300], dtype=np.uint16)
    return np.concatenate([bits, pow2])


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_dequant_exhaustive_codes_vs_rational(fmt):
    scales = _scale_set(fmt, 600, 11 if fmt == "f16" else 12)
    S = scales.size
    # layout: K = 256 rows (16 q values x 16 z values), one group per row
    qz = np.array([(q, z) for q in range(16) for z in range(16)], dtype=np.uint8)
    q = np.repeat(qz[:, 0:1], S, axis=1)                # [256, S]
    z = np.repeat(qz[:, 1:2], S, axis=1)                # group = 1 -> zeros [256, S]
    s = np.repeat(scales[None, :], 256, axis=0)
    with np.errstate(over="ignore"):
        got = oracle.act_bits_to_f64(oracle.dequant_bits(q, s, z, 1, fmt), fmt)
    sval = oracle.act_bits_to_f64(scales, fmt)
    for i, (qq, zz) in enumerate(qz):
        want = [round_exact(Fraction(float(sv)) * (int(qq) - int(zz)), fmt) for sv in sval]
        assert np.array_equal(got[i], np.array(want)), (qq, zz)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_q_equal_zero_point_gives_exact_zero(fmt):
    rng = np.random.default_rng(3)
    K, N, G = 256, 64, 128
    z = rng.integers(0, 16, size=(K // G, N), dtype=np.uint8)
    q = np.repeat(z, G, axis=0)
    s = rng.integers(0x0400, 0x3000, size=(K // G, N), dtype=np.uint16)
    w = oracle.act_bits_to_f64(oracle.dequant_bits(q, s, z, G, fmt), fmt)
    assert np.all(w == 0.0)


def test_symmetric_equals_asymmetric_with_zero_eight():
    rng = np.random.default_rng(5)
    K, N, G = 128, 64, 64
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    s = rng.integers(0x0400, 0x3000, size=(K // G, N), dtype=np.uint16)
    w_sym = oracle.dequant_bits(q, s, None, G, "f16")
    w_asym = oracle.dequant_bits(q, s, np.full((K // G, N), 8, np.uint8), G, "f16")
    assert np.array_equal(w_sym, w_asym)


def test_group_broadcast_and_sign():
    # one column, two groups: scale 0.5 then 2.0, zero 3 then 12
    q = np.array([[0], [3], [15], [12]], dtype=np.uint8)
    s = oracle.rne_f16_bits(np.array([[0.5], [2.0]]))
    z = np.array([[3], [12]], dtype=np.uint8)
    w = oracle.act_bits_to_f64(oracle.dequant_bits(q, s, z, 2, "f16"), "f16")
    assert w.ravel().tolist() == [-1.5, 0.0, 6.0, 0.0]


def test_dequant_rejects_bad_shapes():
    q = np.zeros((100, 64), np.uint8)
    with pytest.raises(ValueError):
        oracle.dequant_bits(q, np.zeros((1, 64), np.uint16), None, 64, "f16")

"""Pins for the oracle's 16-bit round-to-nearest-even casts.

The casts are checked against (a) fixed bit patterns from the IEEE 754
binary16 / bfloat16 definitions (tests/golden/fp16_bf16_rne.txt) and (b) an
exact rational-arithmetic rounding written here from the definition of
round-to-nearest-even.  The dequant step of the method ("I2F scaling",
TurboMind paper, pith.science review, Figure 6) rounds once to 16 bits, so
these casts carry the bit-exactness of the whole dequant oracle.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

FORMATS = {"f16": (11, -14, 15), "bf16": (8, -126, 127)}  # precision, emin, emax


def round_exact(x: Fraction, fmt: str) -> float:
    """Nearest-even rounding of an exact rational into ``fmt`` (inf on overflow)."""
    p, emin, emax = FORMATS[fmt]
    if x == 0:
        return 0.0
    sign = -1.0 if x < 0 else 1.0
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - (p - 1))
    m = a / ulp
    fl = m.numerator // m.denominator
    r = m - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = fl * ulp
    if v >= Fraction(2) ** (emax + 1):
        return sign * math.inf
    return sign * float(v)


def _decode(bits, fmt):
    return oracle.act_bits_to_f64(np.asarray(bits, dtype=np.uint16), fmt)


def _golden_rows():
    rows = []
    with open(os.path.join(HERE, "golden", "fp16_bf16_rne.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v, f16, bf16 = (s.strip() for s in line.split("|"))
            rows.append((v, int(f16, 16), int(bf16, 16)))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_golden_bit_patterns(row):
    expr, f16, bf16 = row
    x = float(eval(expr, {"__builtins__": {}}))  # fixture holds plain arithmetic
    with np.errstate(over="ignore"):
        assert int(oracle.rne_f16_bits(np.array([x]))[0]) == f16
    assert int(oracle.rne_bf16_bits(np.array([x]))[0]) == bf16


def test_decode_known_patterns():
    assert _decode([0x3C00], "f16")[0] == 1.0
    assert _decode([0x7BFF], "f16")[0] == 65504.0
    assert _decode([0x0001], "f16")[0] == 2.0 ** -24
    assert _decode([0x3F80], "bf16")[0] == 1.0
    assert _decode([0xC040], "bf16")[0] == -3.0
    assert _decode([0x0001], "bf16")[0] == 2.0 ** -133


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_rne_matches_exact_rational_rounding(fmt):
    rng = np.random.default_rng(7)
    # float32-representable values over a wide exponent range, both signs,
    # plus values sitting exactly on rounding ties of the target format
    mant = rng.integers(1, 2 ** 24, size=3000)
    exps = rng.integers(-40 if fmt == "f16" else -140, 17, size=3000)
    vals = [float(Fraction(int(m)) * Fraction(2) ** int(e)) * (1 if i % 2 else -1)
            for i, (m, e) in enumerate(zip(mant, exps))]
    p = FORMATS[fmt][0]
    for k in range(1, 200):
        vals.append(float(1 + Fraction(2 * k + 1, 2 ** p)))      # exact ties near 1
        vals.append(float(Fraction(2 * k + 1, 2 ** 25)))          # f16 subnormal ties
    vals = [v for v in vals if np.float32(v) == v]
    x = np.array(vals, dtype=np.float64)
    with np.errstate(over="ignore"):
        bits = oracle.rne_f16_bits(x) if fmt == "f16" else oracle.rne_bf16_bits(x)
    got = _decode(bits, fmt)
    want = np.array([round_exact(Fraction(v), fmt) for v in vals])
    assert np.array_equal(got, want)


def test_bf16_rejects_non_binary32_inputs():
    with pytest.raises(ValueError):
        oracle.rne_bf16_bits(np.array([1.0 + 2.0 ** -30]))

"""Pins for the oracle GEMM C_ref = A @ W (float64) and its tolerance check.

The pages state the GEMM pipeline computes a mixed-precision matrix multiply
of fp16/bf16 activations with dequantized int4 weights (TurboMind paper,
arXiv abstract; pith.science review, Figure 9: MMA on dequantized
fragments).  Pinned by brute force (correctly rounded sums with math.fsum),
one-hot rows, and an integer-arithmetic textbook reduction.
"""

import math

import numpy as np
import pytest

import oracle
from w4a16_gemm_gb300 import synth


def _brute(a_bits, w_bits, fmt):
    A = oracle.act_bits_to_f64(a_bits, fmt)
    W = oracle.act_bits_to_f64(w_bits, fmt)
    M, K = A.shape
    N = W.shape[1]
    out = np.empty((M, N))
    for m in range(M):
        for n in range(N):
            out[m, n] = math.fsum(float(A[m, k]) * float(W[k, n]) for k in range(K))
    return out


@pytest.mark.parametrize("fmt,sym,G", [("f16", False, 128), ("bf16", False, 128), ("f16", True, 64)])
def test_gemm_vs_bruteforce(fmt, sym, G):
    qw, a = synth.random_problem(1, 3, 256, 64, G, fmt, sym)
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, G, fmt)
    c = oracle.gemm_ref(a, w, fmt)
    cb = _brute(a, w, fmt)
    assert np.allclose(c, cb, rtol=1e-12, atol=1e-12 * np.abs(cb).max())


def test_one_hot_rows_reproduce_weight_rows():
    qw, _ = synth.random_problem(2, 1, 256, 64)
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16")
    ks = [0, 1, 127, 128, 255]
    a = np.zeros((len(ks), 256), np.uint16)
    for i, k in enumerate(ks):
        a[i, k] = 0x3C00  # 1.0
    c = oracle.gemm_ref(a, w, "f16")
    W = oracle.act_bits_to_f64(w, "f16")
    for i, k in enumerate(ks):
        assert np.array_equal(c[i], W[k])


def test_textbook_integer_reduction():
    """C = sum_g s_g * (A (Q - Z))_g with integer A and short scales, in int64."""
    rng = np.random.default_rng(9)
    M, K, N, G = 4, 256, 64, 128
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = rng.integers(0, 16, size=(K // G, N), dtype=np.uint8)
    # scales with <= 7 significant bits: m * 2^e, m in [64, 127]
    m = rng.integers(64, 128, size=(K // G, N))
    e = rng.integers(-14, -8, size=(K // G, N))
    s_val = m.astype(np.float64) * np.exp2(e)
    s = oracle.rne_f16_bits(s_val)
    assert np.array_equal(oracle.f16_bits_to_f64(s), s_val)
    a_int = rng.integers(-8, 9, size=(M, K))
    a = oracle.rne_f16_bits(a_int.astype(np.float64))
    w = oracle.dequant_bits(q, s, z, G, "f16")
    assert np.array_equal(oracle.f16_bits_to_f64(w),
                          np.repeat(s_val, G, 0) * (q.astype(np.int64) - np.repeat(z, G, 0)))
    c = oracle.gemm_ref(a, w, "f16")
    qz = q.astype(np.int64) - np.repeat(z.astype(np.int64), G, axis=0)
    want = np.zeros((M, N), dtype=object)
    from fractions import Fraction
    for g in range(K // G):
        part = a_int[:, g * G:(g + 1) * G] @ qz[g * G:(g + 1) * G]   # exact int64
        for i in range(M):
            for j in range(N):
                want[i, j] += Fraction(float(s_val[g, j])) * int(part[i, j])
    want = np.array([[float(x) for x in row] for row in want])
    assert np.array_equal(c, want)


def test_tolerance_detects_planted_mistakes():
    qw, a = synth.random_problem(3, 4, 256, 128)
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16")
    c = oracle.gemm_ref(a, w, "f16")
    c16 = oracle.f16_bits_to_f64(oracle.rne_f16_bits(c))
    assert oracle.tolerance_ok(c16, c)                       # output rounding passes
    # a wrong zero point in one group
    z2 = qw.zeros.copy()
    z2[1, 5] = (z2[1, 5] + 1) % 16
    c_bad = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, z2, 128, "f16"), "f16")
    assert not oracle.tolerance_ok(c_bad, c)
    # a dropped group
    q2 = qw.q.copy()
    q2[128:] = np.repeat(qw.zeros[1:2], 128, axis=0)
    c_bad = oracle.gemm_ref(a, oracle.dequant_bits(q2, qw.scales, qw.zeros, 128, "f16"), "f16")
    assert not oracle.tolerance_ok(c_bad, c)
    # transposed activations (rows swapped)
    assert not oracle.tolerance_ok(c[::-1], c)


def test_rms_and_ratio():
    c = np.array([[3.0, -4.0]])
    assert oracle.rms(c) == pytest.approx(math.sqrt(12.5))
    assert oracle.max_err_ratio(c, c) == 0.0
    assert oracle.max_err_ratio(np.zeros((0, 2)), np.zeros((0, 2))) == 0.0

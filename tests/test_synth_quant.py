"""Invariants of the synthetic RTN quantizer (the stand-in for AWQ/GPTQ inputs)."""

import numpy as np
import pytest

import oracle
from w4a16_gemm_gb300 import synth


@pytest.mark.parametrize("fmt,sym,G", [("f16", False, 128), ("bf16", False, 128), ("f16", True, 64)])
def test_quantizer_invariants(fmt, sym, G):
    rng = np.random.default_rng(21)
    K, N = 512, 96
    w = rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.02)
    qw = synth.quantize_rtn(w, G, fmt, sym)
    assert qw.q.dtype == np.uint8 and qw.q.max() <= 15
    s = oracle.act_bits_to_f64(qw.scales, fmt)
    assert np.all(s > 0)
    deq = oracle.act_bits_to_f64(oracle.dequant_bits(qw.q, qw.scales, qw.zeros, G, fmt), fmt)
    sfull = np.repeat(s, G, 0)
    if sym:
        assert qw.zeros is None
        assert qw.q.min() >= 1                      # rint(x/s) in [-7, 7]
    else:
        assert qw.zeros.max() <= 15
        # the group minimum maps to code 0 unless the zero point clamped
        g = w.reshape(K // G, G, N)
        argmin = np.argmin(g, axis=1)
        qmin = qw.q.reshape(K // G, G, N)[np.arange(K // G)[:, None], argmin, np.arange(N)[None]]
        assert np.all(qmin <= 1)
    # reconstruction error <= s/2 plus the 16-bit rounding of the product
    ulp = np.abs(deq) * (2.0 ** -10 if fmt == "f16" else 2.0 ** -7)
    assert np.all(np.abs(deq - w) <= sfull * 0.5 * (1 + 1e-3) + ulp + 1e-12)


def test_degenerate_group_is_exact_zero():
    w = np.zeros((128, 64), np.float32)
    w[:, 3] = 0.25
    qw = synth.quantize_rtn(w, 128, "f16", False)
    deq = oracle.act_bits_to_f64(oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16"), "f16")
    assert np.all(deq[:, :3] == 0) and np.all(deq[:, 4:] == 0)


def test_workload_seeds_are_stable():
    a1 = synth.activations("tiny", 0, 1)
    a2 = synth.activations("tiny", 0, 1)
    assert np.array_equal(a1, a2)
    qw = synth.weight("tiny", 0)
    assert qw.q.shape == (256, 256) and qw.zeros.shape == (2, 256)
    a = synth.activations("sym_g64", 0, 2)
    assert a.shape == (2, 5120)
    av = oracle.f16_bits_to_f64(a)
    assert np.abs(av).max() <= 64

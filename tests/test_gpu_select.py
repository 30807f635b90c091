"""Variant selection (tm_select): the built-in rule for shapes nobody tuned,
the row-bucket key of the tuned table, and the TM_VARIANT override.

The pages give no selection rule; the built-in one follows the measured
crossovers between the kernels: the register-MMA decode kernel for small row
counts, the tcgen05 decode kernel up to 64 rows, the tcgen05 kernel beyond.
"""

import json
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest
import torch

import oracle
from tests._util import c_values, gemm_poisoned, packed_from
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _fresh_weight(N=1920, K=2048):
    # a shape no other test tunes, so the table has no entry for it
    qw, _ = synth.random_problem(77, 1, K, N)
    return qw, packed_from(qw)


def test_untuned_small_m_runs_a_decode_kernel():
    qw, W = _fresh_weight()
    for M in (1, 2, 3, 4, 8, 12, 16):
        v = binding.select(W, M)
        assert v["kernel"] in ("decode_mma", "gemv", "tc_decode"), (M, v)
    for M in (100, 300, 2048):
        assert binding.select(W, M)["kernel"] == "tc", M
    # the default variants run and match the oracle
    for M in (2, 12, 40):
        a = synth.random_problem(78 + M, M, qw.K, qw.N)[1]
        C = gemm_poisoned(binding.acts_to_device(a, torch.float16), W)
        torch.cuda.synchronize()
        c_ref = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16"), "f16")
        assert oracle.max_err_ratio(c_values(C), c_ref) <= 1.0, M


def test_tuned_entry_covers_its_row_bucket():
    """A table entry measured at M applies to every M of the same power-of-two
    bucket and to no other bucket."""
    qw, W = _fresh_weight(N=2176)
    line = {"N": W.N, "K": W.K, "group": 128, "dtype": 0, "sym": 0, "M": 6, "kernel": 1,
            "block_m": 8, "split_k": 3, "dq_warps": 0, "us": 1.0}
    fd, path = tempfile.mkstemp(suffix=".jsonl")
    with os.fdopen(fd, "w") as f:
        f.write(json.dumps(line) + "\n")
    try:
        assert binding.lib().tm_tune_load(path.encode()) == binding.TM_OK
    finally:
        os.unlink(path)
    for M in (5, 6, 7, 8):
        v = binding.select(W, M)
        assert v["kernel"] == "gemv" and v["split_k"] == 3, (M, v)
    for M in (4, 9):
        assert binding.select(W, M) != binding.select(W, 6), M


def test_tune_picks_a_variant_that_runs():
    qw, W = _fresh_weight(N=2304)
    best = binding.tune(W, [3, 24])
    assert [b["kernel"] for b in best]
    assert binding.select(W, 3) == best[0] and binding.select(W, 4) == best[0]
    assert binding.select(W, 24) == best[1]
    for M in (3, 24):
        a = synth.random_problem(90 + M, M, qw.K, qw.N)[1]
        C = gemm_poisoned(binding.acts_to_device(a, torch.float16), W)
        torch.cuda.synchronize()
        c_ref = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16"), "f16")
        assert oracle.max_err_ratio(c_values(C), c_ref) <= 1.0, M


def test_variant_override_from_the_environment():
    """TM_VARIANT forces a variant wherever it can run (read once per process)."""
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from tests._util import packed_from\n"
        "from w4a16_gemm_gb300 import binding, synth\n"
        "qw, _ = synth.random_problem(79, 1, 2048, 1920)\n"
        "W = packed_from(qw)\n"
        "print(binding.select(W, 4)['kernel'], binding.select(W, 4)['split_k'], binding.select(W, 100)['kernel'])\n"
    ) % ROOT
    env = dict(os.environ, TM_VARIANT="gemv:0:5:0")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    k4, s4, k100 = out.stdout.split()
    assert (k4, s4) == ("gemv", "5")
    assert k100 == "tc"           # the GEMV cannot run 100 rows: regular selection

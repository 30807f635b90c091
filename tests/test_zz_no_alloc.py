"""The GEMM entry point for callers that cannot allocate device memory.

tm_gemm_w4a16_noalloc serves applications that own all GPU memory through
their own pool allocator: its split-K scratch is a fixed static device array
of the library instead of a workspace allocated on demand.  These tests call
it through the C ABI and compare it, within the GEMM tolerance used
throughout the test-suite, with tm_gemm_w4a16_ex running the same variant on
the same inputs, on two calls in a row (the scratch keeps the previous call's
contents), and with the oracle.

Each kernel family is exercised explicitly: the test loads a selection table
(tm_tune_load) that maps its own shapes to the family under test, so the
result does not depend on which tests ran before.  The file is collected
last, so that a run stopping at the first failure has run every other test.
"""

import json
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
from tests._util import TORCH_DT, c_values, packed_from
from w4a16_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TOL = 1e-2
STATIC_WS_BYTES = 8 << 20
STATIC_COUNTERS = 16384

KERNEL_ID = {"gemv": 1, "tc": 2, "tc_decode": 3, "decode_mma": 4}


def _noalloc(A, W, out):
    st = torch.cuda.current_stream().cuda_stream
    M, K = A.shape
    return binding.lib().tm_gemm_w4a16_noalloc(A.data_ptr(), W.handle, out.data_ptr(), M, W.N, K, st)


def _force_variant(W, M, cfg):
    """Makes tm_gemm_w4a16 (and the no-alloc entry point) select cfg for this
    weight's shape at this M, through a loaded selection table."""
    line = {"N": W.N, "K": W.K, "group": W.group, "dtype": 0 if W.dtype == torch.float16 else 1,
            "sym": int(W.symmetric), "M": M, "kernel": KERNEL_ID[cfg["kernel"]],
            "block_m": cfg.get("block_m", 0), "split_k": cfg.get("split_k", 1),
            "dq_warps": cfg.get("dq_warps", 0), "us": 0.0}
    fd, path = tempfile.mkstemp(suffix=".jsonl")
    with os.fdopen(fd, "w") as f:
        f.write(json.dumps(line) + "\n")
    try:
        assert binding.lib().tm_tune_load(path.encode()) == binding.TM_OK
    finally:
        os.unlink(path)
    got = binding.select(W, M)
    assert got["kernel"] == cfg["kernel"], (got, cfg)


def _needed_scratch(W, M, cfg):
    """(bytes of fp32 partials, arrival counters) the variant uses; (0, 0)
    without a split."""
    KB = W.K // 64
    if cfg["kernel"] == "tc_decode":
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        plan = binding.decode_plan(M, W.N, W.K, cfg["block_m"], sms)
        if plan["partial_slots"] <= 1:
            return 0, 0
        return plan["tiles"] * plan["partial_slots"] * 128 * cfg["block_m"] * 4, plan["tiles"]
    if cfg["kernel"] == "decode_mma" and cfg.get("dq_warps", 0) == 1:
        return 0, 0          # cluster split-K: partials stay in shared memory
    if cfg["kernel"] == "decode_mma":
        # persistent stream-K grid: CTAs per SM x SMs over (tile, group) units;
        # contributors of a tile = CTAs whose ranges meet its units
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        cps = binding.select(W, M)["split_k"]          # CTAs per SM, clamped to what fits
        GR, T = W.K // W.group, W.N // 128
        U = T * GR
        G = max(1, min(U, cps * sms))
        begin = lambda c: c * U // G
        def owner(u):
            c = u * G // U
            while c + 1 < G and begin(c + 1) <= u:
                c += 1
            while c > 0 and begin(c) > u:
                c -= 1
            return c
        slots = max(owner((t + 1) * GR - 1) - owner(t * GR) + 1 for t in range(T))
        return (0, 0) if slots <= 1 else (T * slots * M * 128 * 4, T)
    gran = 1
    if cfg["kernel"] == "tc":
        gran = 4 if cfg["block_m"] <= 16 else 2 if cfg["block_m"] <= 64 else 1
    per = -(-KB // cfg.get("split_k", 1))
    per = -(-per // gran) * gran
    splits = -(-KB // per)
    if splits == 1:
        return 0, 0
    counters = W.N // 64 if cfg["kernel"] == "gemv" else (W.N // 128) * (-(-M // cfg["block_m"]))
    return splits * M * W.N * 4, counters


# (M, K, N, dtype, variant): every kernel family, with and without split-K
CASES = [
    (4, 4096, 1152, "f16", dict(kernel="gemv", split_k=4)),
    (1, 2048, 640, "bf16", dict(kernel="gemv", split_k=1)),
    (7, 4096, 1152, "bf16", dict(kernel="gemv", split_k=4, dq_warps=1)),
    (16, 2048, 640, "f16", dict(kernel="gemv", split_k=2, dq_warps=1)),
    (16, 14336, 1152, "f16", dict(kernel="decode_mma", split_k=2)),
    (3, 1024, 640, "bf16", dict(kernel="decode_mma", split_k=1)),
    (9, 4096, 1152, "f16", dict(kernel="decode_mma", split_k=6, dq_warps=1)),
    (2, 8192, 1152, "bf16", dict(kernel="decode_mma", split_k=1, dq_warps=16)),
    (12, 4096, 640, "f16", dict(kernel="decode_mma", split_k=2, dq_warps=8)),
    (16, 4096, 1152, "f16", dict(kernel="tc_decode", block_m=16, dq_warps=8)),
    (40, 2048, 640, "f16", dict(kernel="tc_decode", block_m=32, dq_warps=4)),
    (300, 1024, 1152, "bf16", dict(kernel="tc", block_m=128, split_k=2, dq_warps=8)),
    (64, 4096, 640, "f16", dict(kernel="tc", block_m=64, split_k=1, dq_warps=8)),
]


@pytest.mark.parametrize("M,K,N,dt,cfg", CASES, ids=lambda x: str(x))
def test_matches_the_allocating_entry_point_twice(M, K, N, dt, cfg):
    qw, a = synth.random_problem(40 + M + K // 64, M, K, N, 128, dt)
    W = packed_from(qw)
    A = binding.acts_to_device(a, TORCH_DT[dt])
    _force_variant(W, M, cfg)
    ws_bytes, counters = _needed_scratch(W, M, cfg)
    assert ws_bytes <= STATIC_WS_BYTES and counters <= STATIC_COUNTERS
    ref = binding.gemm(A, W, config=cfg)
    torch.cuda.synchronize()
    c_ref = c_values(ref)
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=TORCH_DT[dt], device="cuda")
        assert _noalloc(A, W, out) == binding.TM_OK, binding.lib().tm_last_error()
        torch.cuda.synchronize()
        c = c_values(out)
        assert np.all(np.isfinite(c))
        assert oracle.max_err_ratio(c, c_ref, rel=TOL) <= 1.0
    assert binding.poll_status() == binding.TM_OK
    w = oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, dt)
    assert oracle.max_err_ratio(c, oracle.gemm_ref(a, w, dt), rel=TOL) <= 1.0


def test_alternating_shapes_reuse_the_scratch():
    """Two problems whose splits differ alternate on the shared scratch: each
    call must clear what it needs and not depend on the previous contents."""
    probs = []
    for (M, K, N, cfg) in ((8, 8192, 640, dict(kernel="decode_mma", split_k=3)),
                           (5, 4096, 1152, dict(kernel="gemv", split_k=3))):
        qw, a = synth.random_problem(60 + M, M, K, N)
        W = packed_from(qw)
        _force_variant(W, M, cfg)
        A = binding.acts_to_device(a, torch.float16)
        c_ref = oracle.gemm_ref(a, oracle.dequant_bits(qw.q, qw.scales, qw.zeros, 128, "f16"), "f16")
        probs.append((W, A, c_ref))
    for i in range(6):
        W, A, c_ref = probs[i % 2]
        out = torch.full((A.shape[0], W.N), float("nan"), dtype=torch.float16, device="cuda")
        assert _noalloc(A, W, out) == binding.TM_OK, binding.lib().tm_last_error()
        torch.cuda.synchronize()
        assert oracle.max_err_ratio(c_values(out), c_ref, rel=TOL) <= 1.0, i
    assert binding.poll_status() == binding.TM_OK


def test_rejects_shapes_beyond_the_static_scratch():
    M, K, N = 64, 14336, 4096
    qw, a = synth.random_problem(50, M, K, N)
    W = packed_from(qw)
    A = binding.acts_to_device(a, torch.float16)
    cfg = dict(kernel="tc", block_m=64, split_k=16, dq_warps=8)    # 16 MiB of partials
    _force_variant(W, M, cfg)
    assert _needed_scratch(W, M, cfg)[0] > STATIC_WS_BYTES
    out = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    assert _noalloc(A, W, out) == binding.TM_ERR_UNSUPPORTED
    assert b"static scratch" in binding.lib().tm_last_error()


def test_m_zero_and_bad_arguments():
    qw, _ = synth.random_problem(51, 1, 256, 256)
    W = packed_from(qw)
    A = torch.zeros((0, 256), dtype=torch.float16, device="cuda")
    out = torch.zeros((0, 256), dtype=torch.float16, device="cuda")
    assert _noalloc(A, W, out) == binding.TM_OK
    st = torch.cuda.current_stream().cuda_stream
    assert binding.lib().tm_gemm_w4a16_noalloc(None, W.handle, None, 1, 256, 256, st) == \
        binding.TM_ERR_INVALID_ARG

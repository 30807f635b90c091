"""Shared helpers of the GPU parity tests (oracle-side sampling and checks)."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from w4a16_gemm_gb300 import binding, synth

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def bits_of(t: torch.Tensor) -> np.ndarray:
    """16-bit tensor -> uint16 bit patterns (numpy)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def packed_from(qw: synth.QuantWeight, device="cuda"):
    p = binding.to_device(qw, device)
    return binding.pack(p.q, p.scales, p.zeros, qw.group)


def sample_indices(n: int, k: int, seed: int, block: int = 128) -> np.ndarray:
    """First/last rows, rows straddling multiples of `block`, and random rows."""
    if n <= k:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    idx = set(range(min(64, n))) | set(range(max(0, n - 64), n))
    for b in range(block, n, block):
        idx.update((b - 1, b))
    idx.update(rng.choice(n, size=min(k, n), replace=False).tolist())
    return np.array(sorted(i for i in idx if 0 <= i < n))


def oracle_sampled(qw: synth.QuantWeight, a_bits: np.ndarray, rows, cols) -> np.ndarray:
    """C_ref[rows][:, cols] from the oracle, dequantizing only the sampled columns."""
    cols = np.asarray(cols)
    z = None if qw.zeros is None else qw.zeros[:, cols]
    w = oracle.dequant_bits(qw.q[:, cols], qw.scales[:, cols], z, qw.group, qw.dtype)
    return oracle.gemm_ref(a_bits[np.asarray(rows)], w, qw.dtype)


def c_values(C: torch.Tensor, rows=None, cols=None) -> np.ndarray:
    c = C.float()
    if rows is not None:
        c = c[torch.as_tensor(np.asarray(rows), device=C.device)]
    if cols is not None:
        c = c[:, torch.as_tensor(np.asarray(cols), device=C.device)]
    return c.cpu().numpy().astype(np.float64)


def gemm_poisoned(A: torch.Tensor, W, config=None) -> torch.Tensor:
    """binding.gemm into an output pre-filled with NaN, so unwritten elements fail."""
    out = torch.full((A.shape[0], W.N), float("nan"), dtype=W.dtype, device=A.device)
    return binding.gemm(A, W, out=out, config=config)

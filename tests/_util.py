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


# Packers into the int32 checkpoint layouts (AWQ, GPTQ), written from the
# column -> nibble direction; oracle/checkpoint.py unpacks nibble -> column.
def awq_pack(q: np.ndarray) -> np.ndarray:
    """uint8 [R, N] -> AWQ int32 [R, N/8]: column offset c goes to nibble POS[c]."""
    POS = (0, 4, 1, 5, 2, 6, 3, 7)
    R, N = q.shape
    w = np.zeros((R, N // 8), dtype=np.int64)
    for c in range(8):
        w |= q[:, c::8].astype(np.int64) << (4 * POS[c])
    return w.astype(np.uint32).astype(np.int32)


def gptq_pack_qweight(q: np.ndarray) -> np.ndarray:
    K, N = q.shape
    w = np.zeros((K // 8, N), dtype=np.int64)
    for r in range(8):
        w |= q[r::8, :].astype(np.int64) << (4 * r)
    return w.astype(np.uint32).astype(np.int32)


def gptq_pack_qzeros(z: np.ndarray, zero_offset: int) -> np.ndarray:
    G, N = z.shape
    stored = z.astype(np.int64) - zero_offset
    w = np.zeros((G, N // 8), dtype=np.int64)
    for c in range(8):
        w |= stored[:, c::8] << (4 * c)
    return w.astype(np.uint32).astype(np.int32)

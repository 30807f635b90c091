"""Oracle for importing int4 checkpoints packed in 32-bit words -- test
infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA path.

The pages evaluate AWQ checkpoints (TurboMind paper, pith.science review,
Figure 11: "Qwen3 8B AWQ") but do not print how such checkpoints store their
codes.  These functions follow the two public packings, read as:

  AWQ ("GEMM" layout)  qweight int32 [K, N/8]; word (k, j) carries the eight
      codes of row k, columns 8j..8j+7; nibble i (bits 4i..4i+3) holds column
      8j + AWQ_COLUMN[i], AWQ_COLUMN = (0, 2, 4, 6, 1, 3, 5, 7).
      qzeros int32 [K/G, N/8] is packed the same way.
  GPTQ  qweight int32 [K/8, N]; word (r, n) carries rows 8r..8r+7 of column
      n, row 8r + i in nibble i.  qzeros int32 [K/G, N/8]; word (g, c)
      carries columns 8c..8c+7 of group g, column 8c + i in nibble i.  The
      original GPTQ files store every zero point minus one: the zero is the
      stored nibble plus `zero_offset` (0 or 1).

Either way the dequantized weight is the method's W = T(s * (q - z)) with
scales [K/G, N]: ``oracle.w4a16.dequant_bits`` applies unchanged.

Parity: pinned by tests/test_oracle_checkpoint.py (hand-computed words and
round trips through packers written independently in the test).
"""

from __future__ import annotations

import numpy as np

AWQ_COLUMN = (0, 2, 4, 6, 1, 3, 5, 7)


def _nibbles(words: np.ndarray) -> np.ndarray:
    """int32 words [..., W] -> their eight nibbles [..., W, 8], nibble i at [..., i]."""
    u = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    return np.stack([(u >> (4 * i)) & 0xF for i in range(8)], axis=-1).astype(np.uint8)


def unpack_awq(packed: np.ndarray) -> np.ndarray:
    """AWQ int32 [R, N/8] (qweight or qzeros) -> uint8 codes [R, N]."""
    nib = _nibbles(packed)                      # [R, N/8, 8], nibble-major
    R, J = packed.shape
    out = np.zeros((R, J, 8), dtype=np.uint8)
    for i, c in enumerate(AWQ_COLUMN):
        out[:, :, c] = nib[:, :, i]
    return out.reshape(R, J * 8)


def unpack_gptq_qweight(packed: np.ndarray) -> np.ndarray:
    """GPTQ qweight int32 [K/8, N] -> uint8 codes [K, N]."""
    nib = _nibbles(packed)                      # [K/8, N, 8]: row 8r + i at nibble i
    R, N = packed.shape
    return np.transpose(nib, (0, 2, 1)).reshape(R * 8, N)


def unpack_gptq_qzeros(packed: np.ndarray, zero_offset: int) -> np.ndarray:
    """GPTQ qzeros int32 [K/G, N/8] -> zero points [K/G, N] (stored nibble + zero_offset)."""
    nib = _nibbles(packed)                      # [G, N/8, 8]: column 8c + i at nibble i
    G, J = packed.shape
    z = nib.reshape(G, J * 8).astype(np.int64) + int(zero_offset)
    if np.any(z > 15):
        raise ValueError("zero point above 15")
    return z.astype(np.uint8)

"""Oracle for decode attention over a low-bit KV cache -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA path.

What it computes (TurboMind paper, pith.science review, Figure 4: the
attention pipeline loads the low-bit KV cache, converts it to 16-bit values
by integer-to-float conversion and scaling, and computes Q K^T and P V;
Figure 10: the cache is consumed in 64-token tiles):

    K[t, d] = RNE_T( ks[t] * (kq[t, d] - kz[t]) )      (per token and KV head)
    V[t, d] = RNE_T( vs[t] * (vq[t, d] - vz[t]) )
    for a query head hq of KV head h = hq // (Hq / Hkv), over t < len:
        S[t]  = sm_scale * sum_d Q[hq, d] * K[t, d]
        P[t]  = exp(S[t] - max S) / sum_t' exp(S[t'] - max S)
        O[hq] = sum_t P[t] * V[t, :]

Readings (the pages print no formula for the cache): the per-token scale
and integer zero of each KV head follow the weights' "I2F conversion and
scaling" (one round-to-nearest-even of the exact product); a sequence of
length 0 attends to nothing and its output is 0.

Layouts (the library's own): Q and O [B, Hq, D]; codes [B, Hkv, L_max, D]
bytes for 8 bits, [B, Hkv, L_max, D/2] for 4 bits with element d in byte
d // 2, the low nibble holding even d; scales [B, Hkv, L_max] 16-bit bit
patterns; zeros [B, Hkv, L_max] bytes.  Tokens at t >= len[b] are ignored.

Everything is float64 after the exact dequantization.

Parity: pinned by tests/test_oracle_attention.py (a pure-Python brute force
with rational dequantization, closed forms for one and two tokens, equal
keys, zero softmax scale, the grouped-query head mapping, the nibble order
and masking of tokens past the length).
"""

from __future__ import annotations

import numpy as np

from .w4a16 import _rne_bits, act_bits_to_f64


def unpack_kv4(codes: np.ndarray) -> np.ndarray:
    """[..., D/2] bytes -> [..., D] 4-bit codes; element d sits in byte d // 2,
    the low nibble for even d, the high nibble for odd d."""
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (2 * c.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = c & 0x0F
    out[..., 1::2] = c >> 4
    return out


def pack_kv4(codes: np.ndarray) -> np.ndarray:
    """Inverse of unpack_kv4: [..., D] codes 0..15 -> [..., D/2] bytes."""
    c = np.asarray(codes, dtype=np.uint8)
    if c.shape[-1] % 2 or c.max(initial=0) > 15:
        raise ValueError("4-bit codes need an even D and values 0..15")
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def kv_dequant_bits(codes: np.ndarray, scale_bits: np.ndarray, zeros: np.ndarray, dtype: str) -> np.ndarray:
    """Cache rows -> 16-bit bit patterns of RNE_T(s[t] * (q[t, d] - z[t])).

    codes [..., T, D] (already unpacked), scale_bits and zeros [..., T].  The
    exact product has at most 11 + 8 significant bits, so float64 holds it and
    the rounding is the only one (pith.science review, Figure 4 text:
    "I2F scaling")."""
    q = np.asarray(codes, dtype=np.float64)
    z = np.asarray(zeros, dtype=np.float64)[..., None]
    s = act_bits_to_f64(np.asarray(scale_bits, dtype=np.uint16), dtype)[..., None]
    with np.errstate(over="ignore", invalid="ignore"):
        return _rne_bits(s * (q - z), dtype)


def attn_decode_ref(q_bits, k_codes, k_scale, k_zero, v_codes, v_scale, v_zero, lens,
                    bits: int, dtype: str, sm_scale: float) -> np.ndarray:
    """O [B, Hq, D] float64 of one decode step (one query token per sequence).

    q_bits [B, Hq, D] 16-bit patterns; k/v codes [B, Hkv, L_max, D] (8 bits)
    or [B, Hkv, L_max, D/2] (4 bits); scales [B, Hkv, L_max] 16-bit patterns;
    zeros [B, Hkv, L_max] bytes; lens [B].  sm_scale is taken as the float32
    value the kernel receives."""
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    q_bits = np.asarray(q_bits, dtype=np.uint16)
    B, Hq, D = q_bits.shape
    Hkv = k_codes.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    grp = Hq // Hkv
    scale = float(np.float32(sm_scale))
    Q = act_bits_to_f64(q_bits, dtype)
    O = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        n = int(lens[b])
        if n == 0:
            continue
        for h in range(Hkv):
            kc, vc = k_codes[b, h, :n], v_codes[b, h, :n]
            if bits == 4:
                kc, vc = unpack_kv4(kc), unpack_kv4(vc)
            K = act_bits_to_f64(kv_dequant_bits(kc, k_scale[b, h, :n], k_zero[b, h, :n], dtype), dtype)
            V = act_bits_to_f64(kv_dequant_bits(vc, v_scale[b, h, :n], v_zero[b, h, :n], dtype), dtype)
            for hq in range(h * grp, (h + 1) * grp):
                s = (K @ Q[b, hq]) * scale
                p = np.exp(s - s.max())
                O[b, hq] = (p @ V) / p.sum()
    return O


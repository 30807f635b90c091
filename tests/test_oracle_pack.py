"""Pins for the oracle's reader/writer of the packed int4 layout.

The packing idea (TurboMind paper, pith.science review, Figures 6 and 7: eight
values per thread fragment, permuted so the runtime load needs no
rearrangement) and the in-word order printed in Figures 23/24 (e7 e5 e3 e1 e6
e4 e2 e0, tests/golden/nibble_order.txt) are checked here, together with the
properties the GPU consumers rely on: each 16-byte chunk holds 32 consecutive
K values of a single column, and pack/unpack are inverse bijections.
"""

import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_nibble_order_matches_pages_figure():
    lines = [l for l in open(os.path.join(HERE, "golden", "nibble_order.txt"))
             if l.startswith("stored:")]
    stored = lines[0].split(":")[1].split()
    # nibble index 7 (most significant) .. 0 holds element stored[i]
    by_pos = {7 - i: int(tok[1:]) for i, tok in enumerate(stored)}
    for e in range(8):
        assert by_pos[oracle.NIBBLE_POS[e]] == e


def test_two_lanes_per_mask():
    """One mask 0x000F000F isolates an (even, odd) pair of consecutive values."""
    q = np.zeros((64, 128), np.uint8)
    q[0:8, 0] = np.arange(1, 9)                  # values 1..8 for k = 0..7 of column 0
    word = int(oracle.pack_ref(q)[:4].view("<u4")[0])
    for pair in range(4):
        lo = (word >> (4 * pair)) & 0xF
        hi = (word >> (16 + 4 * pair)) & 0xF
        assert (lo, hi) == (2 * pair + 1, 2 * pair + 2)


@pytest.mark.parametrize("K,N", [(64, 128), (128, 256), (256, 128), (192, 384)])
def test_roundtrip_random(K, N):
    rng = np.random.default_rng(K * 1000 + N)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    p = oracle.pack_ref(q)
    assert p.dtype == np.uint8 and p.size == K * N // 2
    assert np.array_equal(oracle.unpack_ref(p, K, N), q)


def test_every_value_at_every_position():
    K, N = 128, 128
    kk, nn = np.meshgrid(np.arange(K), np.arange(N), indexing="ij")
    for shift in range(16):
        q = ((kk * 7 + nn * 3 + shift) % 16).astype(np.uint8)
        assert np.array_equal(oracle.unpack_ref(oracle.pack_ref(q), K, N), q)


def test_one_hot_is_a_single_nibble():
    K, N = 128, 128
    rng = np.random.default_rng(0)
    for _ in range(50):
        k, n = int(rng.integers(K)), int(rng.integers(N))
        q = np.zeros((K, N), np.uint8)
        q[k, n] = 0xA
        p = oracle.pack_ref(q)
        nz = np.nonzero(p)[0]
        assert nz.size == 1
        assert p[nz[0]] in (0x0A, 0xA0)


def test_sixteen_byte_chunks_hold_32_consecutive_k_of_one_column():
    K, N = 128, 128
    kk, nn = np.meshgrid(np.arange(K), np.arange(N), indexing="ij")
    # encode (k, n) into two passes of nibbles to locate every value
    locs = {}
    for name, val in (("k_lo", kk % 16), ("k_hi", kk // 16), ("n_lo", nn % 16), ("n_hi", nn // 16)):
        p = oracle.pack_ref(val.astype(np.uint8))
        words = p.view("<u4")
        nib = np.stack([(words >> (4 * oracle.NIBBLE_POS[e])) & 0xF for e in range(8)], 1)
        locs[name] = nib                               # [words, e]
    k_of = locs["k_lo"] + 16 * locs["k_hi"]
    n_of = locs["n_lo"] + 16 * locs["n_hi"]
    chunks_k = k_of.reshape(-1, 32)                    # 4 words x 8 values per 16 B
    chunks_n = n_of.reshape(-1, 32)
    assert np.all(chunks_n == chunks_n[:, :1])         # one column per chunk
    assert np.all(np.diff(chunks_k, axis=1) == 1)      # consecutive K, ascending
    assert np.all(chunks_k[:, 0] % 32 == 0)
    # every (k, n) appears exactly once
    flat = (k_of * N + n_of).ravel()
    assert np.array_equal(np.sort(flat), np.arange(K * N))


def test_zero_pack_roundtrip():
    rng = np.random.default_rng(4)
    z = rng.integers(0, 16, size=(8, 256), dtype=np.uint8)
    zp = oracle.pack_zeros_ref(z)
    assert zp.shape == (8 * 128,)
    assert np.array_equal(oracle.unpack_zeros_ref(zp, 8, 256), z)
    assert zp[0] == (z[0, 0] | (z[0, 1] << 4))
    assert zp[64] == (z[1, 0] | (z[1, 1] << 4))          # next group row of tile 0
    assert zp[8 * 64] == (z[0, 128] | (z[0, 129] << 4))  # first row of tile 1


def test_scale_pack_roundtrip_and_tile_order():
    rng = np.random.default_rng(5)
    s = rng.integers(0, 0x7C00, size=(6, 384), dtype=np.uint16)
    sp = oracle.pack_scales_ref(s)
    assert np.array_equal(oracle.unpack_scales_ref(sp, 6, 384), s)
    # one tile's scales for consecutive groups are contiguous
    assert np.array_equal(sp[128:256], s[1, 0:128])
    assert np.array_equal(sp[6 * 128:7 * 128], s[0, 128:256])


def test_tile_blocks_are_contiguous_in_k():
    """A 128-column tile's consecutive 64-K blocks follow each other (4 KB apart)."""
    K, N = 256, 256
    kk, nn = np.meshgrid(np.arange(K), np.arange(N), indexing="ij")
    p = oracle.pack_ref(((kk // 64) + 4 * (nn // 128)).astype(np.uint8))
    words = p.view("<u4").reshape(-1, 1024)                  # 4 KB blocks
    block_val = words & 0xF                                   # value e0 of each word
    assert np.all(block_val == block_val[:, :1])
    assert block_val[:, 0].tolist() == [0, 1, 2, 3, 4, 5, 6, 7]


def test_pack_rejects_bad_input():
    with pytest.raises(ValueError):
        oracle.pack_ref(np.full((64, 64), 16, np.uint8))
    with pytest.raises(ValueError):
        oracle.pack_ref(np.zeros((64, 64), np.uint8))

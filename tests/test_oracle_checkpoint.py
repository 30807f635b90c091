"""Pins of the checkpoint-import oracle (oracle/checkpoint.py): words whose
unpacking is worked out by hand, and round trips through packers written
here from the opposite direction (column -> nibble position instead of
nibble -> column), so that a swapped permutation, a transposed packing or a
dropped zero offset fails."""

import numpy as np
import pytest

from oracle import checkpoint as ck
from tests._util import awq_pack, gptq_pack_qweight, gptq_pack_qzeros


def _i32(x):
    return np.array(x, dtype=np.uint32).astype(np.int32)


def test_awq_word_by_hand():
    # nibbles 0..7 hold the values 0..7; nibble i is column (0,2,4,6,1,3,5,7)[i]
    q = ck.unpack_awq(_i32([[0x76543210]]))
    assert q.tolist() == [[0, 4, 1, 5, 2, 6, 3, 7]]
    # a word of one code: 0xF in nibble 4 is column 1
    assert ck.unpack_awq(_i32([[0x000F0000]])).tolist() == [[0, 15, 0, 0, 0, 0, 0, 0]]


def test_gptq_words_by_hand():
    # qweight: rows 0..7 of column 0 hold 0..7 (row i in nibble i); column 1 is 0xF... in row 7
    q = ck.unpack_gptq_qweight(_i32([[0x76543210, 0xF0000000]]))
    assert q[:, 0].tolist() == list(range(8)) and q[:, 1].tolist() == [0] * 7 + [15]
    # qzeros: column i in nibble i, plus the offset
    assert ck.unpack_gptq_qzeros(_i32([[0x76543210]]), 0).tolist() == [list(range(8))]
    assert ck.unpack_gptq_qzeros(_i32([[0xEDCBA987]]), 1).tolist() == [list(range(8, 16))]
    with pytest.raises(ValueError):
        ck.unpack_gptq_qzeros(_i32([[0xF0000000]]), 1)


@pytest.mark.parametrize("seed", [0, 1])
def test_round_trips(seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 16, size=(64, 256), dtype=np.uint8)
    assert np.array_equal(ck.unpack_awq(awq_pack(q)), q)
    assert np.array_equal(ck.unpack_gptq_qweight(gptq_pack_qweight(q)), q)
    z = rng.integers(1, 16, size=(4, 256), dtype=np.uint8)
    assert np.array_equal(ck.unpack_gptq_qzeros(gptq_pack_qzeros(z, 1), 1), z)
    assert np.array_equal(ck.unpack_gptq_qzeros(gptq_pack_qzeros(z, 0), 0), z)
    # the two layouts are different: AWQ unpacking of a GPTQ-packed row differs
    assert not np.array_equal(ck.unpack_awq(gptq_pack_qzeros(z, 0)), z)

"""Host-side model of the decode-attention kernel's work split (no GPU).

The kernel scans the sequence lengths into a per-sequence prefix of unit
counts, hands units out by ticket in sequence-major order (sequence, chunk,
KV head), and maps a ticket back with a binary search over the prefix.  A
unit covers chunk c of the sequence: tiles [c * ct, c * ct + ntile) of 64
tokens; a sequence of length 0 keeps one unit with no tiles (its zero
output).  This model restates those rules and checks, for random lengths and
chunk sizes, that every (sequence, KV head) pair sees every token exactly
once, that tickets map back to the unit they were made from, and that the
chunk count the last arriver merges matches the units of that pair.
"""

import bisect

import numpy as np
import pytest

TT = 64


def clamp(n, L_max):
    return 0 if n < 0 else min(n, L_max)


def units_of(n, ct, Hkv):
    ctok = ct * TT
    return Hkv * (1 if n == 0 else (n + ctok - 1) // ctok)


def prefix(lens, ct, Hkv):
    pref = [0]
    for n in lens:
        pref.append(pref[-1] + units_of(n, ct, Hkv))
    return pref


def unit(u, pref, lens, ct, Hkv):
    """Ticket u -> (b, h, c, t0, ntile, nch), as the producer lane derives it."""
    b = bisect.bisect_right(pref, u) - 1           # the last b with pref[b] <= u
    n = lens[b]
    ctok = ct * TT
    nch = 1 if n == 0 else (n + ctok - 1) // ctok
    r = u - pref[b]
    c, h = r // Hkv, r % Hkv
    t0 = c * ctok
    ntile = 0 if n == 0 else min(ct, (n - t0 + TT - 1) // TT)
    return b, h, c, t0, ntile, nch


@pytest.mark.parametrize("seed", range(20))
def test_every_token_once_and_tickets_round_trip(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    Hkv = int(rng.choice([1, 2, 8]))
    L_max = 64 * int(rng.integers(1, 40))
    ct = int(rng.integers(1, L_max // 64 + 2))
    raw = rng.integers(-5, L_max + 100, size=B)
    raw[rng.random(B) < 0.2] = 0
    lens = [clamp(int(n), L_max) for n in raw]
    pref = prefix(lens, ct, Hkv)
    seen = {}
    chunks = {}
    for u in range(pref[-1]):
        b, h, c, t0, ntile, nch = unit(u, pref, lens, ct, Hkv)
        assert 0 <= b < B and 0 <= h < Hkv and 0 <= c < nch
        assert pref[b] + c * Hkv + h == u                       # round trip
        chunks.setdefault((b, h), set()).add(c)
        assert chunks[(b, h)] <= set(range(nch))
        for tt in range(ntile):
            first = t0 + tt * TT
            assert first < lens[b] and first + TT <= L_max     # tiles start inside the sequence and the cache
            for tok in range(first, min(first + TT, lens[b])):
                key = (b, h, tok)
                assert key not in seen, key
                seen[key] = u
    for b in range(B):
        for h in range(Hkv):
            assert all((b, h, tok) in seen for tok in range(lens[b]))
            n_units = units_of(lens[b], ct, Hkv) // Hkv
            assert chunks[(b, h)] == set(range(n_units))         # the merge sees every chunk
    assert len(seen) == Hkv * sum(lens)


def test_empty_sequences_keep_one_unit_per_head():
    lens, ct, Hkv = [0, 0, 130], 1, 2
    pref = prefix(lens, ct, Hkv)
    assert pref == [0, 2, 4, 4 + 2 * 3]
    got = [unit(u, pref, lens, ct, Hkv)[:5] for u in range(pref[-1])]
    assert got[:4] == [(0, 0, 0, 0, 0), (0, 1, 0, 0, 0), (1, 0, 0, 0, 0), (1, 1, 0, 0, 0)]
    assert [g[4] for g in got[4:]] == [1, 1, 1, 1, 1, 1]        # 130 tokens: three one-tile chunks


def test_last_partial_tile():
    # 200 tokens in chunks of 2 tiles: chunk 0 = tiles 0-1, chunk 1 = tiles 2-3 (the last partial)
    pref = prefix([200], 2, 1)
    assert [unit(u, pref, [200], 2, 1)[3:5] for u in range(pref[-1])] == [(0, 2), (128, 2)]

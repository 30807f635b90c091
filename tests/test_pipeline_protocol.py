"""Randomized model of the tcgen05 kernel's mbarrier pipeline (CPU).

The kernel overlaps copies, dequantization and MMAs -- the Blackwell
restatement of the parallel MMA-dequantization of the TurboMind paper
(pith.science review, Figure 9).  Its barriers are waited on by phase
parity, which cannot tell phase c from phase c-2, so each wait is correct
only if the waiter already knows that the previous phase completed.  This
model runs the producer, the MMA thread and every dequant warp as independent
agents under random schedules, with copies that land out of order and MMAs
that retire in order, and checks that no agent ever reads a shared-memory
slot or TMEM slot holding the wrong data.  Every variant the library accepts
(tm_tc_pipeline) must be clean; a layout that breaks the rule must be caught.
"""

import random

import pytest


class _Bar:
    def __init__(self, count):
        self.count, self.arr, self.tx, self.phase = count, 0, 0, 0

    def arrive(self):
        self.arr += 1
        self._check()

    def expect_tx(self, b):
        self.tx += b
        self.arrive()

    def complete_tx(self, b):
        self.tx -= b
        self._check()

    def _check(self):
        assert self.arr <= self.count, "too many arrivals in one phase"
        if self.arr == self.count and self.tx == 0:
            self.phase += 1
            self.arr = 0

    def try_wait(self, parity):        # true iff the phase of that parity has completed
        return (self.phase & 1) != parity


def simulate(S, TS, KBS, WG, nkb, seed, max_steps=200_000):
    rnd = random.Random(seed)
    nst = (nkb + KBS - 1) // KBS
    full = [_Bar(1) for _ in range(S)]
    empty = [_Bar(1 + 4) for _ in range(S)]
    afull = [_Bar(4) for _ in range(TS)]
    aempty = [_Bar(1) for _ in range(TS)]
    accum = _Bar(1)
    smem = [None] * S
    tmem = [[None] * 4 for _ in range(TS)]
    events, errors = [], []
    clock = [0, 0]            # now, last MMA retirement time

    def at(t, fn):
        events.append((t, rnd.random(), fn))

    def producer():
        for j in range(nst):
            s = j % S
            if j >= S:
                while not empty[s].try_wait(((j // S) & 1) ^ 1):
                    yield
            full[s].expect_tx(1)
            smem[s] = None

            def land(s=s, j=j):
                smem[s] = j
                full[s].complete_tx(1)
            at(clock[0] + rnd.randint(3, 80), land)     # copies land out of order
            yield

    def mma():
        for j in range(nst):
            s = j % S
            while not full[s].try_wait((j // S) & 1):
                yield
            if smem[s] != j:
                errors.append(f"MMA: smem slot {s} holds {smem[s]}, wanted stage {j}")
            for b in range(min(KBS, nkb - j * KBS)):
                i = j * KBS + b
                t = i % TS
                while not afull[t].try_wait((i // TS) & 1):
                    yield
                if any(tmem[t][q] != i for q in range(4)):
                    errors.append(f"MMA: TMEM slot {t} not ready for block {i}")
                clock[1] = max(clock[1], clock[0]) + rnd.randint(1, 25)   # in-order retirement

                def retire(t=t, i=i, s=s, j=j):
                    if any(tmem[t][q] != i for q in range(4)) or smem[s] != j:
                        errors.append(f"operands of block {i} overwritten before it retired")
                    aempty[t].arrive()
                at(clock[1], retire)
                yield
            at(clock[1] + 0.1, lambda s=s: empty[s].arrive())
        at(clock[1] + 0.2, accum.arrive)

    def warp(g, q):
        for j in range(g, nst, WG):
            s = j % S
            while not full[s].try_wait((j // S) & 1):
                yield
            nb = min(KBS, nkb - j * KBS)
            for b in range(nb):
                i = j * KBS + b
                t = i % TS
                if i >= TS:
                    while not aempty[t].try_wait(((i // TS) & 1) ^ 1):
                        yield
                if smem[s] != j:
                    errors.append(f"warp {g}.{q}: smem slot {s} holds {smem[s]}, wanted stage {j}")
                if b == nb - 1:
                    empty[s].arrive()
                yield
                tmem[t][q] = None          # tcgen05.st in flight
                yield
                tmem[t][q] = i
                afull[t].arrive()
        while not accum.try_wait(0):
            yield

    agents = [producer(), mma()] + [warp(g, q) for g in range(WG) for q in range(4)]
    alive = list(range(len(agents)))
    for _ in range(max_steps):
        events.sort()
        while events and events[0][0] <= clock[0]:
            events.pop(0)[2]()
        if errors:
            return errors[0]
        if not alive and not events:
            return None
        if alive and rnd.random() < 0.8:
            k = rnd.choice(alive)
            try:
                next(agents[k])
            except StopIteration:
                alive.remove(k)
        else:
            clock[0] += 1
    return "did not finish"


def _library_variants():
    from w4a16_gemm_gb300 import binding, build

    build.build()
    out = []
    for bm in (16, 32, 64, 128, 256):
        for dq in (4, 8, 16):
            info = binding.tc_pipeline(bm, dq)
            out.append((bm, dq, info))
    return out


@pytest.fixture(scope="module")
def variants():
    return _library_variants()


def test_model_catches_a_layout_that_breaks_the_rule():
    # 5 shared-memory slots shared round-robin by 4 warpgroups
    failures = [simulate(5, 8, 1, 4, nkb=40, seed=s) for s in range(30)]
    assert any(f is not None for f in failures)


def test_every_accepted_variant_is_race_free(variants):
    for bm, dq, info in variants:
        if not info["legal"]:
            continue
        for seed in range(40):
            nkb = 37 if seed % 2 else 64
            err = simulate(info["stages"], info["tmem_slots"], info["kblocks_per_stage"], dq // 4,
                           nkb=nkb, seed=seed)
            assert err is None, (bm, dq, info, seed, err)


def test_rule_matches_the_library(variants):
    for bm, dq, info in variants:
        wg = dq // 4
        rule = (info["stages"] % wg == 0 and
                info["tmem_slots"] >= (wg - 1) * info["kblocks_per_stage"] + 1)
        assert info["legal"] == rule, (bm, dq, info)

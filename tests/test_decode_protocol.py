"""CPU checks of the tcgen05 decode kernel's stream-K plan and barrier protocol.

The decode kernel splits the (tile, 256-K stage) units of a GEMM evenly over
a persistent grid; tiles cut between CTAs are finished by the last CTA to
arrive.  Its roles (weight producer, activation producer, one MMA issuer and
one dequant warpgroup per ring, an epilogue warpgroup) meet at mbarriers that
are waited on by phase parity, which cannot tell phase c from phase c-2.  The
model below runs every role as an independent agent under random schedules,
with copies that land out of order and each issuer's MMAs retiring in order,
using the ring sizes the library reports (tm_tc_decode_pipeline), and checks
that no agent reads a slot holding the wrong data, that no operand or
accumulator is overwritten before it is consumed, and that every tile
segment's accumulator holds exactly its blocks when the epilogue reads it.
"""

import random

import pytest

WKB = 4          # 64-K blocks per stage


def _cta_range(c, U, G):
    return c * U // G, (c + 1) * U // G


def test_plan_partitions_every_unit_once():
    from w4a16_gemm_gb300 import binding

    for (M, N, K, bm, sms) in [(16, 28672, 4096, 16, 152), (1, 4096, 4096, 16, 152),
                               (40, 128, 1216, 16, 152), (64, 4096, 14336, 64, 148),
                               (16, 256, 8192, 16, 152), (4, 256, 256, 16, 152)]:
        plan = binding.decode_plan(M, N, K, bm, sms)
        S = (K // 64 + WKB - 1) // WKB
        T = (N // 128) * ((M + bm - 1) // bm)
        U = T * S
        G = plan["grid"]
        assert plan["tiles"] == T and G == min(sms, U)
        covered = []
        max_contrib = 1
        for c in range(G):
            lo, hi = _cta_range(c, U, G)
            assert hi > lo                       # no idle CTA
            covered.extend(range(lo, hi))
        assert covered == list(range(U))
        for t in range(T):
            owners = {c for c in range(G) for u in range(*_cta_range(c, U, G)) if u // S == t}
            assert owners == set(range(min(owners), max(owners) + 1))
            max_contrib = max(max_contrib, len(owners))
        assert plan["partial_slots"] == max_contrib, (M, N, K, bm, plan, max_contrib)


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


def simulate_decode(WST, ASW, TSW, DQ, stages, seed, max_steps=400_000):
    """stages: the CTA's stages in order, as (tile, blocks).  Returns None or
    the first error found."""
    rnd = random.Random(seed)
    n = len(stages)
    wfull = [_Bar(1) for _ in range(WST)]
    wempty = [_Bar(4) for _ in range(WST)]
    afull = [_Bar(1) for _ in range(DQ * ASW)]
    aempty = [_Bar(1) for _ in range(DQ * ASW)]
    tfull = [[_Bar(4) for _ in range(TSW)] for _ in range(DQ)]
    kfree = [[_Bar(1) for _ in range(TSW)] for _ in range(DQ)]
    accfull = [[_Bar(1), _Bar(1)] for _ in range(DQ)]
    accempty = [[_Bar(4), _Bar(4)] for _ in range(DQ)]
    smem_w = [None] * WST
    smem_a = [None] * (DQ * ASW)
    tmem = [[[None] * 4 for _ in range(TSW)] for _ in range(DQ)]
    acc = [[None, None] for _ in range(DQ)]
    acc_read = [[True, True] for _ in range(DQ)]
    events, errors = [], []
    clock = [0]
    ret = [0] * DQ                 # each issuer's last MMA retirement (in order)

    def at(t, fn):
        events.append((t, rnd.random(), fn))

    def wait(bar, parity):
        while not bar.try_wait(parity):
            yield

    def w_producer():
        for j in range(n):
            s = j % WST
            if j >= WST:
                yield from wait(wempty[s], ((j // WST) & 1) ^ 1)
            wfull[s].expect_tx(1)
            smem_w[s] = None

            def land(s=s, j=j):
                smem_w[s] = j
                wfull[s].complete_tx(1)
            at(clock[0] + rnd.randint(3, 80), land)     # copies land out of order
            yield

    def a_producer():
        for j in range(n):
            w, cs = j % DQ, j // DQ
            s = w * ASW + cs % ASW
            if cs >= ASW:
                yield from wait(aempty[s], ((cs // ASW) & 1) ^ 1)
            afull[s].expect_tx(1)
            smem_a[s] = None

            def land(s=s, j=j):
                smem_a[s] = j
                afull[s].complete_tx(1)
            at(clock[0] + rnd.randint(3, 80), land)
            yield

    def mma(w, j, b, slot, as_, buf, first, after=None):
        ret[w] = max(ret[w], clock[0]) + rnd.randint(1, 25)

        def retire():
            if any(tmem[w][slot][q] != (j, b) for q in range(4)) or smem_a[as_] != j:
                errors.append(f"issuer {w}: operands of block ({j},{b}) overwritten before it retired")
            if first:
                if not acc_read[w][buf]:
                    errors.append(f"issuer {w}: accumulator {buf} reused before the epilogue read it")
                acc[w][buf] = []
                acc_read[w][buf] = False
            acc[w][buf].append((j, b))
            kfree[w][slot].arrive()
            if after is not None:
                after()
        at(ret[w], retire)

    def issuer(w):
        c, e, t_cur = 0, -1, None
        mine = list(range(w, n, DQ))
        for cs, j in enumerate(mine):
            t, nb = stages[j]
            first = False
            if t != t_cur:
                t_cur, e, first = t, e + 1, True
                if e >= 2:
                    yield from wait(accempty[w][e & 1], ((e >> 1) & 1) ^ 1)
            as_ = w * ASW + cs % ASW
            yield from wait(afull[as_], (cs // ASW) & 1)
            if smem_a[as_] != j:
                errors.append(f"issuer {w}: activation slot {as_} holds {smem_a[as_]}, wanted {j}")
            last_of_seg = cs + 1 == len(mine) or stages[mine[cs + 1]][0] != t
            buf = e & 1

            def end_of_stage(as_=as_, buf=buf, last_of_seg=last_of_seg):
                aempty[as_].arrive()
                if last_of_seg:
                    accfull[w][buf].arrive()
            groups = [(0, 2), (2, 2)] if nb == WKB else [(b, 1) for b in range(nb)]
            for gi, (b0, cnt) in enumerate(groups):
                cl = c + cnt - 1                    # the group's last block covers it
                yield from wait(tfull[w][cl % TSW], (cl // TSW) & 1)
                for h in range(cnt):
                    slot = (c + h) % TSW
                    if any(tmem[w][slot][q] != (j, b0 + h) for q in range(4)):
                        errors.append(f"issuer {w}: TMEM slot {slot} not ready for ({j},{b0 + h})")
                    is_last = gi == len(groups) - 1 and h == cnt - 1
                    mma(w, j, b0 + h, slot, as_, buf, first and gi == 0 and h == 0,
                        end_of_stage if is_last else None)
                c += cnt
                yield

    def dequant_warp(w, q):
        c = 0
        for j in range(w, n, DQ):
            s = j % WST
            yield from wait(wfull[s], (j // WST) & 1)
            t, nb = stages[j]
            groups = [(0, 2), (2, 2)] if nb == WKB else [(b, 1) for b in range(nb)]
            for gi, (b0, cnt) in enumerate(groups):
                if smem_w[s] != j:
                    errors.append(f"warp {w}.{q}: weight slot {s} holds {smem_w[s]}, wanted {j}")
                cl = c + cnt - 1                # the later block's slot free covers both
                if cl >= TSW:
                    yield from wait(kfree[w][cl % TSW], ((cl // TSW) & 1) ^ 1)
                yield
                for h in range(cnt):
                    tmem[w][(c + h) % TSW][q] = None      # tcgen05.st in flight
                yield
                for h in range(cnt):
                    tmem[w][(c + h) % TSW][q] = (j, b0 + h)
                for h in range(cnt):
                    tfull[w][(c + h) % TSW].arrive()
                if gi == len(groups) - 1:
                    if smem_w[s] != j:
                        errors.append(f"warp {w}.{q}: weight slot {s} overwritten while in use")
                    wempty[s].arrive()          # the stage's data has been used
                c += cnt

    def epilogue():
        e_of = [-1] * DQ
        jseg = 0
        while jseg < n:
            t = stages[jseg][0]
            jend = jseg
            while jend < n and stages[jend][0] == t:
                jend += 1
            for qq in range(min(jend - jseg, DQ)):
                w = (jseg + qq) % DQ
                e_of[w] += 1
                e = e_of[w]
                buf = e & 1
                yield from wait(accfull[w][buf], (e >> 1) & 1)
                want = [(j, b) for j in range(jseg, jend) if j % DQ == w for b in range(stages[j][1])]
                if acc[w][buf] != want:
                    errors.append(f"epilogue: tile {t} warpgroup {w} accumulator holds {acc[w][buf]}")
                acc_read[w][buf] = True
                yield
                for _ in range(4):
                    accempty[w][buf].arrive()
            jseg = jend

    agents = ([w_producer(), a_producer(), epilogue()] + [issuer(w) for w in range(DQ)] +
              [dequant_warp(w, q) for w in range(DQ) for q in range(4)])
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


def _stage_list(rnd):
    """A CTA's stages from a random stream-K range: tile boundaries, ragged
    last stages (K not a multiple of 256) and a random start."""
    S = rnd.randint(2, 6)
    KB = S * WKB - rnd.randint(0, WKB - 1)
    u0 = rnd.randint(0, 3 * S)
    nloc = rnd.randint(1, 28)
    return [((u // S), min(WKB, KB - (u % S) * WKB)) for u in range(u0, u0 + nloc)]


@pytest.fixture(scope="module")
def decode_variants():
    from w4a16_gemm_gb300 import binding, build

    build.build()
    return [(bm, dq, binding.tc_decode_pipeline(bm, dq))
            for bm in (16, 32, 64) for dq in (4, 8, 12, 16)]


def test_every_accepted_decode_variant_is_race_free(decode_variants):
    rnd = random.Random(1)
    checked = 0
    for bm, dq, info in decode_variants:
        if not info["legal"]:
            continue
        for seed in range(25):
            stages = _stage_list(rnd)
            err = simulate_decode(info["weight_stages"], info["act_stages_per_wg"],
                                  info["tmem_slots_per_wg"], dq // 4, stages, seed)
            assert err is None, (bm, dq, info, stages, seed, err)
            checked += 1
    assert checked >= 200


def test_decode_model_catches_a_ring_too_small_for_a_pair():
    # one TMEM slot per warpgroup cannot hold a block pair: the model must
    # report the overwrite or a stall (the library refuses such variants)
    failures = [simulate_decode(4, 2, 1, 2, [(t // 3, WKB) for t in range(12)], seed=s)
                for s in range(10)]
    assert any(f is not None for f in failures)


def test_decode_model_catches_a_weight_ring_shared_across_warpgroups():
    # 5 weight slots over 2 warpgroups: a warp may poll a slot whose previous
    # phase belonged to the other warpgroup and take phase c - 2 for c
    rnd = random.Random(3)
    failures = [simulate_decode(5, 2, 4, 2, _stage_list(rnd), seed=s) for s in range(200)]
    assert any(f is not None and "weight slot" in f for f in failures)

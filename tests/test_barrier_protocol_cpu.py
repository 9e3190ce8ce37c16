"""The two linear kernels' barrier protocols, simulated on the host under
random schedules.

Every role of a CTA (producer, decode or compute warps, MMA warp, epilogue) is
a generator that runs the same index arithmetic as the kernel and waits on
simulated mbarriers with the kernel's parities. An mbarrier completes a phase
when its expected arrivals and transaction bytes are in; a parity wait passes
while the barrier's current phase has the other parity, which is how
`mbarrier.try_wait.parity` behaves. Copies land in any order; tensor-core work
(the tcgen05 kernel's MMAs and their commits) completes at random later
times, in issue order for each issuing warp and in any order between the
two. Every buffer carries a tag naming the unit, half-unit or
segment whose data it holds, and every read and every asynchronous MMA checks
the tag: a wait that passed on a stale phase, a stage refilled while still
being read, or an accumulator reused too early fails the test. A schedule that
leaves work undone with nothing runnable is a deadlock and fails too.

A planted fault (a stage count that is not a multiple of the consumers, the
kind of assignment that once let a wait run two phases ahead) must be caught.
"""

import random

import pytest

from test_pipeline_cpu import SegmentOrder, ranges


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.phase = name, count, count, 0, 0

    def arrive(self, n=1):
        assert self.pending >= n, "%s: more arrivals than the phase expects" % self.name
        self.pending -= n
        self._complete()

    def arrive_expect_tx(self, nbytes):
        self.tx += nbytes
        self.arrive()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        assert self.tx >= 0, "%s: bytes beyond the expected count" % self.name
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.phase & 1) != parity


class Sim:
    """Random scheduler over role generators and asynchronous events."""

    def __init__(self, rng):
        self.rng = rng
        self.roles = []          # [generator, pending wait or None]
        self.copies = []         # copies in flight: callables, land in any order
        self.tensor = [[], []]   # per issuing warp: callables, each queue completes in order

    def add(self, gen):
        self.roles.append([gen, None])

    def run(self, max_steps=2_000_000):
        for _ in range(max_steps):
            ready = [r for r in self.roles if r[1] is None or r[1][0].passes(r[1][1])]
            queues = [t for t in self.tensor if t]
            events = len(self.copies) + len(queues)
            if not ready and not events:
                if self.roles:
                    names = [r[1][0].name for r in self.roles if r[1] is not None]
                    raise AssertionError("deadlock: roles wait on %s" % names)
                return
            pick = self.rng.randrange(len(ready) + events)
            if pick < len(ready):
                role = ready[pick]
                try:
                    role[1] = next(role[0])
                except StopIteration:
                    self.roles.remove(role)
            elif pick - len(ready) < len(self.copies):
                self.copies.pop(pick - len(ready))()
            else:
                queues[pick - len(ready) - len(self.copies)].pop(0)()
        raise AssertionError("schedule did not finish")


def wait(bar, parity):
    """Yield point of a role: resumes once `bar` passes `parity`."""
    return (bar, parity)


# --------------------------------------------------------------------------
# The tcgen05 kernel: producer, WG decode warpgroups, MMA warp, epilogue.

def run_tc(order, S, H, rng, ACC=2, plant=None, WG=4, SW=None):
    """The tcgen05 kernel: a weights producer and an xr producer, each
    refilling its part of a unit's stages (one copy per unit of H half-units
    where the ring allows) once that part's readers are done (the decode
    warpgroups for the weights, the MMAs for xr); WG decode warpgroups
    (half-unit q to warpgroup q mod WG), each with one A buffer whose uses
    go to whichever chain the half-unit belongs to, signalled through four
    full barriers (use j on barrier j mod 4); one MMA warp per chain (units
    at even / odd processing positions), each issuing its chain's MMAs in
    order, a whole unit's at once (after waiting for all its half-units)
    where one copy brings the unit; ACC accumulator sets alternating between
    segments.
    `plant` names a fault to plant: "w_early" refills a stage's weights
    without waiting for the decode, "x_early" its xr slice without waiting
    for the MMAs, "no_dempty" starts a segment without waiting for the
    readout of its accumulator set, "a_early" decodes into an A buffer
    without waiting for the MMAs that read it before, "one_afull" signals
    every use of an A buffer on a single full barrier, "two_units" has an
    MMA warp wait for two of its chain's units before issuing either (a
    warpgroup's next half-unit then waits on MMAs that wait on it)."""
    sim = Sim(rng)
    n_half = order.n_units * H
    CG = H if (S >= 8 and S % (WG * H // (H if WG % H == 0 else 1)) == 0) else 1
    SU = S // CG             # copy slots: the barriers go by copies
    SW = S if SW is None else SW   # the weights ring may be deeper than the xr ring
    SUW = SW // CG
    wfull = [Bar("wfull%d" % s, 1) for s in range(SUW)]
    wempty = [Bar("wempty%d" % s, 4 * CG) for s in range(SUW)]
    xfull = [Bar("xfull%d" % s, 1) for s in range(SU)]
    xempty = [Bar("xempty%d" % s, CG) for s in range(SU)]
    AF = 1 if plant == "one_afull" else 4  # full barriers per warpgroup: use j on barrier j % AF
    afull = [[Bar("afull%d.%d" % (g, b), 4) for b in range(AF)] for g in range(WG)]
    aempty = [Bar("aempty%d" % g, 1) for g in range(WG)]
    dfull = [Bar("dfull%d" % d, 2) for d in range(ACC)]
    dempty = [Bar("dempty%d" % d, 4) for d in range(ACC)]
    wtag = [None] * SW       # half-unit whose weights a stage holds
    xtag = [None] * S        # half-unit whose xr slice a stage holds
    abuf = [None] * WG  # half-unit whose decoded weights a warpgroup's A buffer holds
    acc = [[None, None] for _ in range(ACC)]  # segment whose sums a chain's accumulator holds

    def producer(full, empty, tag, wait_empty, SU):
        for u in range(n_half // CG):
            us = u % SU
            if u >= SU and wait_empty:
                yield wait(empty[us], ((u // SU) - 1) & 1)
            full[us].arrive_expect_tx(1)

            def land(us=us, u=u):
                for h in range(CG):
                    tag[us * CG + h] = u * CG + h
                full[us].complete_tx(1)
            sim.copies.append(land)

    def decode(wg):
        j = 0
        while WG * j + wg < n_half:
            q = WG * j + wg
            s = q % SW
            yield wait(wfull[s // CG], (q // SW) & 1)
            if j >= 1 and plant != "a_early":
                yield wait(aempty[wg], (j - 1) & 1)
            assert wtag[s] == q, "decode of %d read stage %d holding %s" % (q, s, wtag[s])
            abuf[wg] = q
            yield None                                    # the decode takes a while
            assert wtag[s] == q, "stage %d refilled while half-unit %d was decoded" % (s, q)
            for _ in range(4):
                wempty[s // CG].arrive()
                afull[wg][j % AF].arrive()
            j += 1

    def segments():
        for sg in range(order.n_seg):
            bb = order.block(sg)
            lo = order.lo(bb)
            yield sg, order.pos(sg, lo), order.hi(bb) - lo

    def mma(ch):
        for sg, P, L in segments():
            d = sg % ACC
            if sg >= ACC and plant != "no_dempty":
                yield wait(dempty[d], ((sg // ACC) - 1) & 1)
            kf = P + ((ch - P) & 1)
            if kf >= P + L:
                dfull[d].arrive()                            # no unit of this chain here
                continue
            # The chain's half-units in groups: every wait of a group first,
            # then its MMAs (a whole unit where one copy brings it). The
            # "two_units" plant groups a unit with the chain's next one.
            ks = list(range(kf, P + L, 2))
            if plant == "two_units":
                groups = [[k * H + h for k in ks[i:i + 2] for h in range(H)] for i in range(0, len(ks), 2)]
            else:
                B = H if CG == H else 1
                groups = [[k * H + h0 + i for i in range(B)] for k in ks for h0 in range(0, H, B)]
            for grp in groups:
                for q in grp:
                    s = q % S
                    assert ((q // H) & 1) == ch
                    if s % CG == 0:                          # the first half-unit of its copy
                        yield wait(xfull[s // CG], (q // S) & 1)
                    jj = q // WG
                    yield wait(afull[q % WG][jj % AF], (jj // AF) & 1)
                for q in grp:
                    s = q % S
                    g = q % WG

                    def execute(q=q, s=s, g=g, sg=sg, d=d, first=(q == kf * H)):
                        assert xtag[s] == q, "MMA of %d found stage %d's xr of %s" % (q, s, xtag[s])
                        assert abuf[g] == q, "MMA of %d found A buffer %d holding %s" % (q, g, abuf[g])
                        if first:
                            acc[d][ch] = sg
                        assert acc[d][ch] == sg, "chain %d MMA of segment %d into sums of %s" % (
                            ch, sg, acc[d][ch])
                        aempty[g].arrive()                   # the two commits after the MMAs
                        xempty[s // CG].arrive()
                    sim.tensor[ch].append(execute)
            sim.tensor[ch].append(dfull[d].arrive)           # commit at the segment's end

    def epilogue():
        for sg, P, L in segments():
            d = sg % ACC
            yield wait(dfull[d], (sg // ACC) & 1)
            has = [L >= 2 or P % 2 == ch for ch in range(2)]
            for ch in range(2):
                if has[ch]:
                    assert acc[d][ch] == sg, "segment %d read chain %d sums of %s" % (sg, ch, acc[d][ch])
            yield None                                    # the readout takes a while
            for ch in range(2):
                if has[ch]:
                    assert acc[d][ch] == sg, "chain %d sums of segment %d overwritten" % (ch, sg)
            for _ in range(4):
                dempty[d].arrive()

    sim.add(producer(wfull, wempty, wtag, plant != "w_early", SUW))
    sim.add(producer(xfull, xempty, xtag, plant != "x_early", SU))
    for wg in range(WG):
        sim.add(decode(wg))
    sim.add(mma(0))
    sim.add(mma(1))
    sim.add(epilogue())
    sim.run()
    assert all(wtag[s] is not None for s in range(min(SW, n_half)))


# --------------------------------------------------------------------------
# The mma.sync kernel: producer, two compute groups, epilogue.

def run_mma(order, S, rng, groups=2):
    sim = Sim(rng)
    n = order.n_units
    full = [Bar("full%d" % s, 1) for s in range(S)]
    empty = [Bar("empty%d" % s, 1) for s in range(S)]   # one arrival per group here (8 warps in the kernel)
    dfull = [Bar("dfull%d" % d, groups) for d in range(2)]
    dempty = [Bar("dempty%d" % d, 1) for d in range(2)]
    stage = [None] * S
    dbuf = [[None] * groups for _ in range(2)]
    prod = []
    for q in range(order.n_seg):
        bb = order.block(q)
        prod.extend(order.u0 + i for i in range(order.lo(bb), order.hi(bb)))

    def producer():
        for k in range(n):
            s = k % S
            if k >= S:
                yield wait(empty[s], ((k // S) - 1) & 1)
            full[s].arrive_expect_tx(1)

            def land(s=s, k=k):
                stage[s] = prod[k]
                full[s].complete_tx(1)
            sim.copies.append(land)

    def compute(cg):
        for sg in range(order.n_seg):
            bb = order.block(sg)
            seg_lo, seg_hi = order.lo(bb), order.hi(bb)
            base = order.pos(sg, seg_lo) - seg_lo
            i = seg_lo + ((cg - base - seg_lo) % groups)
            while i < seg_hi:
                k = base + i
                s = k % S
                yield wait(full[s], (k // S) & 1)
                assert stage[s] == order.u0 + i, "group %d read stage %d holding unit %s, wanted %d" % (
                    cg, s, stage[s], order.u0 + i)
                yield None
                assert stage[s] == order.u0 + i, "stage %d refilled during its unit" % s
                empty[s].arrive()
                i += groups
            d = sg & 1
            if sg >= 2:
                yield wait(dempty[d], ((sg >> 1) - 1) & 1)
            dbuf[d][cg] = sg
            dfull[d].arrive()

    def epilogue():
        for sg in range(order.n_seg):
            d = sg & 1
            yield wait(dfull[d], (sg >> 1) & 1)
            assert dbuf[d] == [sg] * groups, "segment %d read sums %s" % (sg, dbuf[d])
            yield None
            assert dbuf[d] == [sg] * groups, "sums of segment %d overwritten" % sg
            dempty[d].arrive()

    sim.add(producer())
    for cg in range(groups):
        sim.add(compute(cg))
    sim.add(epilogue())
    sim.run()


def cta_orders(seed, n):
    rng = random.Random(seed)
    for _ in range(n):
        ub = rng.choice([1, 2, 3, 5, 10, 20])
        units = ub * rng.randint(1, 12)
        ctas = min(units, rng.choice([1, 2, 3, 5, 7]))
        c = rng.randrange(ctas)
        u0, u1 = ranges(units, ctas)[c]
        yield SegmentOrder(u0, u1, ub)


# (xr stages, half-units per unit, accumulator sets, decode warpgroups,
# weights stages): every row-slot class the kernel is built for (2..8 bits;
# 16, 32, 64, 128 row slots; one or two half-units per unit; the list
# `tc_rings` of the pipeline test derives), then others.
REAL_CLASSES = [(4, 1, 1, 4, 4), (4, 1, 1, 4, 8), (4, 1, 1, 4, 12), (4, 1, 1, 4, 20), (4, 1, 2, 4, 8),
                (4, 1, 2, 4, 12), (4, 2, 1, 4, 4), (6, 1, 2, 5, 10), (6, 1, 2, 6, 12), (8, 1, 2, 4, 8),
                (8, 2, 2, 4, 8), (10, 1, 2, 5, 10), (10, 2, 2, 5, 10), (12, 1, 2, 6, 12), (12, 2, 2, 6, 12),
                (15, 1, 2, 5, 15)]


@pytest.mark.parametrize("S,H,ACC,WG,SW", REAL_CLASSES + [(16, 2, 2, 4, 16), (12, 2, 2, 4, 12), (20, 2, 2, 5, 20),
                                                         (10, 2, 2, 5, 20)])
def test_tc_kernel_protocol_under_random_schedules(S, H, ACC, WG, SW):
    rng = random.Random(100 * S + 10 * H + ACC + 1000 * WG + 7 * SW)
    for order in cta_orders(S * 4 + H + WG + SW, 60):
        for _ in range(3):
            run_tc(order, S, H, rng, ACC, WG=WG, SW=SW)


@pytest.mark.parametrize("plant", ["w_early", "x_early", "no_dempty", "a_early", "one_afull", "two_units"])
def test_tc_planted_faults_are_caught(plant):
    """A producer that refills its part of a stage without waiting for that
    part's reader, or a chain that starts a segment in an accumulator set
    the epilogue may still be reading, must fail some schedule."""
    rng = random.Random(21)
    failures = 0
    for order in cta_orders(21, 60):
        for _ in range(5):
            try:
                run_tc(order, 10, 2, rng, 1 if plant == "no_dempty" else 2, plant=plant, WG=5)
            except AssertionError:
                failures += 1
    assert failures > 0


@pytest.mark.parametrize("S", [4, 6, 8, 10, 12])
def test_mma_kernel_protocol_under_random_schedules(S):
    rng = random.Random(S)
    for order in cta_orders(50 + S, 80):
        for _ in range(3):
            run_mma(order, S, rng)


def test_planted_fault_is_caught():
    """A stage count that is not a multiple of the decode warpgroups: a
    stage's previous half-unit went to another warpgroup, so a wait can pass
    on the wrong phase. Some schedule must fail."""
    rng = random.Random(7)
    failures = 0
    for order in cta_orders(7, 400):
        for _ in range(5):
            try:
                run_tc(order, 6, 2, rng, 2, WG=4)
            except AssertionError:
                failures += 1
    assert failures > 0


def test_xr_ring_off_the_chain_period_is_caught():
    """Control: six xr slots of single half-units at two half-units per unit
    (a chain period of four) with five warpgroups: a slot's consecutive uses
    alternate chains. Some schedule must fail."""
    failures = 0
    for seed in range(60):
        rng = random.Random(seed)
        for order in cta_orders(seed + 3000, 60):
            try:
                run_tc(order, 6, 2, rng, 1, WG=5, SW=5)
            except AssertionError:
                failures += 1
        if failures:
            break
    assert failures > 0


def test_odd_xr_ring_below_two_stages_per_warpgroup_is_caught():
    """Control for the xr ring rule: five xr slots of single half-units with
    five warpgroups (what the 8-bit, 32-row-slot class had) let the MMA warp
    of half-unit q + 5 test the slot's barrier before the other chain's copy
    of q landed. Some schedule must fail."""
    failures = 0
    for seed in range(40):
        rng = random.Random(seed)
        for order in cta_orders(seed + 1000, 60):
            try:
                run_tc(order, 5, 1, rng, 2, WG=5, SW=10)
            except AssertionError:
                failures += 1
        if failures:
            break
    assert failures > 0


def test_planted_fault_in_the_mma_kernel_is_caught():
    """An odd stage count in the mma.sync kernel: unit k and unit k - S go to
    different groups."""
    rng = random.Random(8)
    failures = 0
    for order in cta_orders(8, 40):
        for _ in range(5):
            try:
                run_mma(order, 5, rng)
            except AssertionError:
                failures += 1
    assert failures > 0

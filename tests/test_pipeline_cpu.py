"""Host-side check of the two linear kernels' stage rings (their index
formulas, restated from the kernels): the order in which a CTA's producer
fills stages is the order its consumers take them, every unit is taken once,
and a stage's previous unit (S positions earlier) was taken by the same
consumer.

The last property keeps every mbarrier wait within one phase of its barrier:
a consumer waits for unit k only after it took unit k - S from the same stage,
and the copy of unit k + S cannot complete before it releases unit k, so the
parity a wait tests can never stand for two phases at once. An earlier stage
assignment without it (an odd stage count, groups chosen by range index) was
safe only while copies landed in issue order."""

import math
import random

import pytest

KIB = 1024


class SegmentOrder:
    """A CTA's units [u0, u1) of the block-major (block, unit) grid, as
    segments of one block each; a range that ends inside a block (shared with
    the next CTA) takes that block first."""

    def __init__(self, u0, u1, ub):
        self.u0, self.ub, self.n_units = u0, ub, u1 - u0
        self.b_first, self.b_last = u0 // ub, (u1 - 1) // ub
        self.n_seg = self.b_last - self.b_first + 1
        self.n_last = self.n_units - self.lo(self.b_last)
        self.rotated = self.n_seg >= 2 and u1 % ub != 0

    def block(self, q):
        if self.rotated:
            return self.b_last if q == 0 else self.b_first + q - 1
        return self.b_first + q

    def lo(self, bb):
        return bb * self.ub - self.u0 if bb * self.ub > self.u0 else 0

    def hi(self, bb):
        return min((bb + 1) * self.ub - self.u0, self.n_units)

    def pos(self, q, seg_lo):
        if self.rotated:
            return 0 if q == 0 else self.n_last + seg_lo
        return seg_lo


def producer_units(o):
    """Unit at each processing position, in the producer's (cursor's) order."""
    out = []
    for q in range(o.n_seg):
        bb = o.block(q)
        out.extend(o.u0 + i for i in range(o.lo(bb), o.hi(bb)))
    return out


def mma_consumers(o, groups=2):
    """The mma.sync kernel: compute group cg takes, in each segment, the units
    at processing positions k = base + i with k % groups == cg, in order.
    Returns {position: (group, unit)}."""
    taken = {}
    for cg in range(groups):
        last = -1
        for q in range(o.n_seg):
            bb = o.block(q)
            seg_lo, seg_hi = o.lo(bb), o.hi(bb)
            base = o.pos(q, seg_lo) - seg_lo
            i = seg_lo + ((cg - base - seg_lo) % groups)
            while i < seg_hi:
                k = base + i
                assert k % groups == cg and k > last
                taken[k] = (cg, o.u0 + i)
                last = k
                i += groups
    return taken


def tc_mma_walk(o, halves):
    """The tcgen05 kernel's MMA warp: half-unit q = k * halves + h of unit
    position k, in its loop order. Returns [(q, unit, h)]."""
    walk = []
    for sg in range(o.n_seg):
        bb = o.block(sg)
        seg_lo, seg_hi = o.lo(bb), o.hi(bb)
        base = o.pos(sg, seg_lo) - seg_lo
        for i in range(seg_lo, seg_hi):
            k = base + i
            for h in range(halves):
                walk.append((k * halves + h, o.u0 + i, h))
    return walk


def mma_stages(bits, ukt, budget=196 * KIB):
    """Stage count of the mma.sync kernel (16 row slots, two groups)."""
    slots = 16
    stage = 256 * bits * ukt + 128 * slots * (ukt // 4)
    dbuf = 2 * 2 * slots * 128 * 4
    fit = (budget - dbuf - 8192 - 1024) // stage
    return min(fit, 12) & ~1


def tc_stages(bits, slots, halves=2, budget=227 * KIB):
    """Stage count, decode warpgroups and half-units per copy of the tcgen05
    kernel's class: six warpgroups at 16 row slots and 4, 6 or 8 bits, five
    otherwise up to 32 row slots, four beyond; the stage count a multiple of
    the warpgroups, and of the half-units of a unit where that still leaves
    8 stages or more (then one copy per unit)."""
    wg = 6 if (slots == 16 and bits in (4, 6, 8)) else (5 if slots <= 32 else 4)
    stage = 256 * bits * 8 + slots * 16 * 8 * 2
    cap = min((budget - 8192 - 2048) // stage, 16)
    step = wg * halves // math.gcd(wg, halves)
    if cap // step * step >= 8:
        return cap // step * step, wg, halves
    return cap // wg * wg, wg, 1


def tc_rings(bits, slots, halves=2, budget=227 * KIB):
    """The tcgen05 kernel's two rings: (xr stages, weights stages, decode
    warpgroups, half-units per copy). The xr ring is the base stage count,
    rounded up to a multiple of the chains' period (2 * halves) below two
    stages per warpgroup;
    where the base leaves fewer than two stages per warpgroup and copies
    bring whole units, the weights ring takes the rest of shared memory, a
    multiple of its step, capped at 24."""
    s, wg, cg = tc_stages(bits, slots, halves, budget)
    wbytes, xbytes = 256 * bits * 8, slots * 16 * 8 * 2
    sx = (s // (2 * halves) + 1) * 2 * halves if (s < 2 * wg and s % (2 * halves)) else s
    step = wg * halves // math.gcd(wg, halves) if cg == halves else wg
    wcap = min((budget - 8192 - 2048 - sx * xbytes) // wbytes, 24)
    sw = wcap // step * step if (s < 2 * wg and cg == halves and wcap // step * step > s) else s
    return sx, sw, wg, cg


def ranges(units, ctas):
    return [(c * units // ctas, (c + 1) * units // ctas) for c in range(ctas)]


def random_shapes(n, seed):
    rng = random.Random(seed)
    for _ in range(n):
        ub = rng.choice([1, 2, 3, 5, 10, 20, 24, 40, 64])
        units = ub * rng.randint(1, 300)
        yield ub, units, min(units, rng.choice([1, 2, 3, 7, 132, 152, 160]))
    # the LM head and wkv at 16- and 8-k-tile units, on 152 SMs
    yield 20, 1010 * 20, 152
    yield 40, 1010 * 40, 152
    yield 24, 200 * 24, 152
    yield 48, 200 * 48, 152


@pytest.mark.parametrize("stages", [4, 6, 8, 10, 12])
def test_mma_kernel_groups_keep_their_stages(stages):
    for ub, units, ctas in random_shapes(300, seed=stages):
        seen = []
        for u0, u1 in ranges(units, ctas):
            o = SegmentOrder(u0, u1, ub)
            prod = producer_units(o)
            taken = mma_consumers(o)
            assert sorted(taken) == list(range(o.n_units))
            for k, (cg, unit) in taken.items():
                assert prod[k] == unit                      # the stage holds the unit its consumer expects
                if k >= stages:
                    assert taken[k - stages][0] == cg       # the stage's previous unit: same group
            seen.extend(prod)
        assert sorted(seen) == list(range(units))


@pytest.mark.parametrize("halves", [1, 2])
def test_tc_kernel_walk_matches_producer(halves):
    for ub, units, ctas in random_shapes(300, seed=10 + halves):
        for u0, u1 in ranges(units, ctas):
            o = SegmentOrder(u0, u1, ub)
            prod = producer_units(o)
            walk = tc_mma_walk(o, halves)
            # The MMA warp takes half-units in the producer's order: q runs
            # 0, 1, 2, ... and half-unit q is half q % halves of the unit at
            # position q // halves.
            assert [q for q, _, _ in walk] == list(range(o.n_units * halves))
            for q, unit, h in walk:
                assert prod[q // halves] == unit and q % halves == h


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_stage_counts_keep_each_stage_with_one_consumer(bits):
    for ukt in ([16, 8] if bits <= 5 else [8]):
        s = mma_stages(bits, ukt)
        assert s >= 4 and s % 2 == 0, (bits, ukt, s)       # two groups, two stages each at least
    for slots in (16, 32, 64, 128):
        for halves in (1, 2):
            s, wg, cg = tc_stages(bits, slots, halves)
            assert s >= wg and s % wg == 0 and s % cg == 0, (bits, slots, s)
            # Half-unit q is decoded by warpgroup q % wg from stage q % s, so
            # the stage's previous half-unit q - s went to the same
            # warpgroup; a copy group's half-units are consecutive.
            for q in range(s, 4 * s):
                assert (q - s) % wg == q % wg
                assert (q - s) // cg % (s // cg) == q // cg % (s // cg)


def test_stage_counts_of_the_measured_classes():
    """The counts the measurements were taken with (4 bits)."""
    assert mma_stages(4, 16) == 6
    assert tc_stages(4, 16) == (12, 6, 2)
    assert tc_stages(2, 16) == (10, 5, 2)
    assert tc_stages(4, 32) == (10, 5, 2)
    assert tc_stages(4, 64) == (8, 4, 2)
    assert tc_stages(4, 128) == (4, 4, 1)


def test_ring_depths_keep_their_waits_within_one_phase():
    for bits in (2, 3, 4, 5, 6, 8):
        for halves in ((2, 1) if bits <= 5 else (1,)):
            for slots in (16, 32, 64, 128):
                sx, sw, wg, cg = tc_rings(bits, slots, halves)
                assert sw % wg == 0 and sw % cg == 0 and sx % cg == 0, (bits, slots, halves)
                # below two stages per warpgroup the xr ring is a multiple of the
                # chains' period, so that a slot's consecutive uses go to one chain
                assert sx >= 2 * wg or sx % (2 * halves) == 0, (bits, slots, halves)
                assert sw * 256 * bits * 8 + sx * slots * 16 * 8 * 2 + 8192 + 2048 <= 227 * KIB


def test_ring_depths_of_the_measured_classes():
    assert tc_rings(4, 16) == (12, 12, 6, 2)
    assert tc_rings(8, 16, 1) == (6, 12, 6, 1)
    assert tc_rings(8, 32, 1) == (6, 10, 5, 1)
    assert tc_rings(6, 64, 1) == (4, 12, 4, 1)
    assert tc_rings(8, 64, 1) == (4, 8, 4, 1)
    assert tc_rings(4, 128) == (4, 4, 4, 1)

"""The fused rotation's hand-over between CTAs, simulated on the host under
random schedules.

tf_rot_in_linear's launch rotates the pass's (row, 128-block) units inside
the linear kernel. Three counters in global memory carry the hand-over:
count 0 hands units out, count 1 counts the units rotated, and count 2 counts
the CTAs done with both. In each CTA, five actors take part:
- the four epilogue warps each ask for units until a request comes back past
  the last one, rotate what they got, and add that to count 1;
- the xr producer waits until count 1 holds every unit, and only then starts
  its copies of xr.
A shared-memory count finds the CTA's last actor, which counts the CTA into
count 2; the CTA that completes count 2 resets all three. Each actor here is
a generator that takes the kernel's steps one atomic at a time, in any order;
CTAs may start late, after others have finished. A step that touches the
counters after the reset, a copy of xr before all its rows are in, or counters
left non-zero at the end fails the test. Two launches run back to back on the
same counters, as consecutive calls do.

Planted faults (the CTA counted in after four actors instead of five, and a
producer that polls the hand-out count instead of the done count) must be
caught.
"""

import random

import pytest


class Launch:
    def __init__(self, sync, ctas, units, fin_needed=5, poll_index=1):
        self.sync, self.ctas, self.units = sync, ctas, units
        self.fin = [0] * ctas
        self.written = set()
        self.reset_done = False
        self.fin_needed = fin_needed
        self.poll_index = poll_index
        self.copies_started = 0

    def touch(self):
        assert not self.reset_done, "a counter touched after the reset"

    def cta_done(self, c):
        self.fin[c] += 1
        if self.fin[c] == self.fin_needed:
            self.touch()
            self.sync[2] += 1
            if self.sync[2] == self.ctas:
                self.sync[0] = self.sync[1] = self.sync[2] = 0
                self.reset_done = True

    def warp(self, c):
        done = 0
        while True:
            self.touch()
            u = self.sync[0]
            self.sync[0] += 1
            yield
            if u >= self.units:
                break
            assert u not in self.written
            self.written.add(u)       # the rotation's stores (then a fence)
            done += 1
            yield
        if done:
            self.touch()
            self.sync[1] += done
            yield
        self.cta_done(c)

    def producer(self, c):
        while True:
            self.touch()
            if self.sync[self.poll_index] >= self.units:
                break
            yield
        assert len(self.written) == self.units, "xr copied before every unit was rotated"
        self.copies_started += 1
        self.cta_done(c)
        yield


def run_launch(sync, ctas, units, rng, late=(), **kw):
    launch = Launch(sync, ctas, units, **kw)
    actors = {}
    for c in range(ctas):
        for w in range(4):
            actors[(c, w)] = launch.warp(c)
        actors[(c, "p")] = launch.producer(c)
    # CTAs in `late` start only once every other CTA has finished (their SM
    # was held by the kernel before).
    waiting = {k: g for k, g in actors.items() if k[0] in late}
    running = {k: g for k, g in actors.items() if k[0] not in late}
    steps = 0
    while running or waiting:
        if not running:
            running, waiting = waiting, {}
        k = rng.choice(list(running))
        try:
            next(running[k])
        except StopIteration:
            del running[k]
        steps += 1
        assert steps < 10 ** 6, "no progress"
    assert launch.copies_started == ctas
    assert launch.written == set(range(units))
    assert sync == [0, 0, 0], "counters left at %s" % sync
    return launch


@pytest.mark.parametrize("ctas,units", [(1, 1), (2, 4), (4, 40), (8, 3), (16, 160), (32, 640)])
@pytest.mark.parametrize("seed", range(6))
def test_every_unit_before_any_copy_and_counters_back_to_zero(ctas, units, seed):
    rng = random.Random(1000 * ctas + units + seed)
    sync = [0, 0, 0]
    for _ in range(2):  # two launches back to back on the same counters
        late = set(rng.sample(range(ctas), k=min(ctas - 1, rng.randint(0, 3)))) if ctas > 1 else set()
        run_launch(sync, ctas, units, rng, late=late)


def test_one_running_cta_rotates_everything():
    """Every CTA but one starts late: the one running does all the units and
    starts its copies; no CTA waits for another to be resident."""
    rng = random.Random(7)
    sync = [0, 0, 0]
    launch = run_launch(sync, 8, 64, rng, late=set(range(1, 8)))
    assert launch.copies_started == 8


def test_reset_after_four_actors_is_caught():
    """Control: counting the CTA in after four actors (forgetting one warp or
    the producer) lets the reset race a late actor."""
    caught = 0
    for seed in range(40):
        rng = random.Random(seed)
        try:
            run_launch([0, 0, 0], 8, 40, rng, fin_needed=4, late={3})
        except AssertionError:
            caught += 1
    assert caught > 0


def test_producer_polling_the_hand_out_count_is_caught():
    """Control: a producer that waits on the count of units handed out (not
    rotated) starts copying rows that are not written yet."""
    caught = 0
    for seed in range(40):
        rng = random.Random(seed)
        try:
            run_launch([0, 0, 0], 8, 40, rng, poll_index=0)
        except AssertionError:
            caught += 1
    assert caught > 0

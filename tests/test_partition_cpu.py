"""Host-side check of the persistent linear's work split (the formulas the
kernel uses, restated): the (output block, 128-input unit) grid cut into one
contiguous range per CTA. Each unit belongs to exactly one CTA, the CTA of a
unit inverts the ranges, a CTA cuts at most its first and last block, and no
two CTAs write the same partial-sum slot for a block."""

import pytest


def range_start(c, units, ctas):
    return c * units // ctas


def cta_of_unit(u, units, ctas):
    return ((u + 1) * ctas - 1) // units


def partial_slot(c, b, units, ctas, ub):
    return 0 if b == range_start(c, units, ctas) // ub else 1


@pytest.mark.parametrize("unit_inputs", [128, 256])
@pytest.mark.parametrize("i_f,o_f,sms", [(5120, 129280, 152), (6144, 25600, 152), (512, 128, 152),
                                         (384, 256, 152), (5120, 129280, 148), (128, 128, 4),
                                         (6144, 128, 152), (1024, 8192, 132)])
def test_partition_covers_each_unit_once(i_f, o_f, sms, unit_inputs):
    if i_f % unit_inputs:
        pytest.skip("unit size does not divide the inputs")
    ub = i_f // unit_inputs
    units = (o_f // 128) * ub
    ctas = min(sms, units)
    owner = {}
    for c in range(ctas):
        u0, u1 = range_start(c, units, ctas), range_start(c + 1, units, ctas)
        assert u1 > u0
        for u in range(u0, u1):
            assert u not in owner
            owner[u] = c
            assert cta_of_unit(u, units, ctas) == c
    assert len(owner) == units
    for b in range(o_f // 128):
        cf = cta_of_unit(b * ub, units, ctas)
        cl = cta_of_unit((b + 1) * ub - 1, units, ctas)
        slots = {(c, partial_slot(c, b, units, ctas, ub)) for c in range(cf, cl + 1)}
        assert len(slots) == cl - cf + 1
        for c in range(cf, cl + 1):
            u0, u1 = range_start(c, units, ctas), range_start(c + 1, units, ctas)
            first_b, last_b = u0 // ub, (u1 - 1) // ub
            assert b in (first_b, last_b) or (first_b < b < last_b and cf == cl)

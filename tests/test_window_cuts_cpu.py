"""The column decode's window cuts against the oracle's trellis states.

At 2, 4, 6 and 8 bits the kernels cut a column's 16 windows out of a few
words with fixed shifts, byte permutes and masks (`decode_col16_b2`, `_b4`,
`_b6`, `_b8` and `load_col_words` in the decode header, restated here). For
random tiles, the 16 states that thread n forms must equal the oracle's states
of stream weights 16n .. 16n + 15 (the direct windows of the bitshift
trellis), for every column n of the tile.
"""

import numpy as np
import pytest

from oracle import exl3 as o

M32 = 0xFFFFFFFF


def funnel_l(lo, hi, sh):
    """Upper 32 bits of (hi:lo) << sh, as CUDA's __funnelshift_l(lo, hi, sh)."""
    return ((((hi << 32) | lo) << (sh & 31)) >> 32) & M32


def hi16(x):
    return x >> 16


def mid16(x):
    return (x >> 8) & 0xFFFF


def lo16(x):
    return x & 0xFFFF


def window16(p, hi, lo):
    """The 16-bit window from bit p (counted from the top) of `hi` on into `lo`."""
    if p == 0:
        return hi16(hi)
    if p == 8:
        return mid16(hi)
    if p == 16:
        return lo16(hi)
    if p < 16:
        return (hi >> (16 - p)) & 0xFFFF
    if p == 24:
        return mid16(funnel_l(lo, hi, 16))
    return funnel_l(lo, hi, p) >> 16


def column_states(w, bits, n):
    w = [int(x) for x in w]
    if bits == 2:
        a, b = w[(n + 15) & 15], w[n]
        x2, x4, x6, m = funnel_l(b, a, 18), funnel_l(b, a, 20), funnel_l(b, a, 22), funnel_l(b, a, 16)
        y2, y4, y6 = (b << 2) & M32, (b << 4) & M32, (b << 6) & M32
        return [hi16(x2), hi16(x4), hi16(x6), mid16(m), mid16(x2), mid16(x4), mid16(x6), hi16(b),
                lo16(x2), lo16(x4), lo16(x6), mid16(b), mid16(y2), mid16(y4), mid16(y6), lo16(b)]
    if bits == 4:
        a, b, c = w[(2 * n + 31) & 31], w[2 * n], w[2 * n + 1]
        p, m, b4 = funnel_l(b, a, 12), funnel_l(b, a, 16), b >> 4
        p2, m2, c4 = funnel_l(c, b, 12), funnel_l(c, b, 16), c >> 4
        return [mid16(p), mid16(m), lo16(p), hi16(b), mid16(b4), mid16(b), lo16(b4), lo16(b),
                mid16(p2), mid16(m2), lo16(p2), hi16(c), mid16(c4), mid16(c), lo16(c4), lo16(c)]
    if bits == 6:
        ww = [w[47 if n == 0 else 3 * n - 1]] + [w[3 * n + j] for j in range(3)]
        out = []
        for j in range(16):
            start = 22 + 6 * j
            k = start // 32
            out.append(window16(start % 32, ww[k], ww[min(k + 1, 3)]))
        return out
    assert bits == 8
    a = w[(4 * n + 63) & 63]
    b, c, d, e = (w[4 * n + j] for j in range(4))
    ab, bc, cd, de = funnel_l(b, a, 16), funnel_l(c, b, 16), funnel_l(d, c, 16), funnel_l(e, d, 16)
    return [mid16(ab), hi16(b), mid16(b), lo16(b), mid16(bc), hi16(c), mid16(c), lo16(c),
            mid16(cd), hi16(d), mid16(d), lo16(d), mid16(de), hi16(e), mid16(e), lo16(e)]


@pytest.mark.parametrize("bits", [2, 4, 6, 8])
def test_window_cuts_match_oracle_states(bits):
    rng = np.random.default_rng(100 + bits)
    for _ in range(40):
        words = rng.integers(0, 2 ** 32, size=8 * bits, dtype=np.uint64).astype(np.uint32)
        states = o.tile_states(words, bits)
        for n in range(16):
            assert column_states(words, bits, n) == [int(v) for v in states[16 * n:16 * n + 16]], (bits, n)


@pytest.mark.parametrize("bits", [2, 4, 6, 8])
def test_a_cut_one_bit_off_is_caught(bits):
    """Control: the same comparison with column n's window 5 cut one bit late
    (the funnel shift or window start one more) must fail for some column."""
    rng = np.random.default_rng(7)
    words = rng.integers(0, 2 ** 32, size=8 * bits, dtype=np.uint64).astype(np.uint32)
    states = o.tile_states(words, bits)
    w = [int(x) for x in words]
    per = 8 * bits
    caught = False
    for n in range(16):
        # the words of the column from its first window's word on, and the
        # window's start counted from that word's top bit, one bit late
        first = (16 * n * bits + bits - 16) % (256 * bits)
        w0, off = first // 32, first % 32
        start = off + 5 * bits + 1
        k = start // 32
        cut = window16(start % 32, w[(w0 + k) % per], w[(w0 + k + 1) % per])
        got = column_states(words, bits, n)
        got[5] = cut
        caught |= got != [int(v) for v in states[16 * n:16 * n + 16]]
    assert caught

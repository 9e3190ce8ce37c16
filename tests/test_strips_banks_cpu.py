"""The strips order against the tcgen05 kernel's shared-memory reads.

A thread decoding column n of a tile reads, for each group of four k-tiles,
the word quads (16 bytes each) of words 2n-1, 2n, 2n+1 at 4 bits and 4n-1 ..
4n+3 at 8 bits (mod the tile's 8 * bits words), at the positions written in
`load_col_quads` (restated here). Those positions must hold exactly those
words in the strips order the oracle defines, and the 128-bit loads of each
eight consecutive threads (one shared-memory wavefront) must fall in eight
distinct 16-byte bank groups.
"""

import pytest

from oracle import exl3 as o


def kernel_positions(bits, n):
    if bits == 4:
        return [16 + ((n + 15) & 15), n, 16 + n]
    return [48 + ((n + 15) & 15)] + [16 * j + n for j in range(4)]


def words_needed(bits, n):
    per = 8 * bits
    step = bits // 2
    first = (step * n - 1) % per
    return [(first + i) % per for i in range(3 if bits == 4 else 5)]


@pytest.mark.parametrize("bits", [4, 8])
def test_positions_hold_the_words_each_thread_decodes(bits):
    pos = o.strips_quad_positions(bits)
    for n in range(16):
        assert [pos[w] for w in words_needed(bits, n)] == kernel_positions(bits, n)


@pytest.mark.parametrize("bits", [4, 8])
def test_each_wavefront_is_free_of_bank_conflicts(bits):
    # A warp covers two tiles (threads 0-15 and 16-31); a tile's quads span
    # 8 * bits * 16 bytes, a multiple of the 128-byte bank period, so the
    # second tile repeats the first one's banks.
    for load in range(3 if bits == 4 else 5):
        for phase in range(2):
            groups = {kernel_positions(bits, n)[load] % 8 for n in range(8 * phase, 8 * phase + 8)}
            assert len(groups) == 8

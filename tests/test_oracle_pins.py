"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself (a value printed on the page, a closed form, an exact
integer identity, an independent brute-force routine), and the planted-fault
checks show that a plausible mistake in the oracle turns a pin red.

Page: "hip exl3: the input rotation and trellis linear for decode rows"
(TensorFold pull request #3314).
"""

import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import exl3 as o
from trellis_quantized_linear_rot_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Independent scalar helpers (plain Python integers, fractions and struct).
# ---------------------------------------------------------------------------
def f16_value(bits):
    """fp16 bit pattern -> exact Fraction (finite values only)."""
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 10) & 0x1F
    m = bits & 0x3FF
    assert e != 0x1F
    if e == 0:
        return sign * Fraction(m, 1 << 24)
    return sign * Fraction(1024 + m, 1 << 10) * (Fraction(2) ** (e - 15))


_POS_F16 = [(f16_value(b), b) for b in range(0x7C00)]   # ascending in value


def nearest_f16_bits(q):
    """Round a Fraction to fp16, ties to even mantissa, overflow to inf."""
    q = Fraction(q)
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    if a >= Fraction(65520):
        return sign | 0x7C00
    lo, hi = 0, len(_POS_F16) - 1
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _POS_F16[mid][0] <= a:
            lo = mid
        else:
            hi = mid
    (vl, bl), (vh, bh) = _POS_F16[lo], _POS_F16[hi]
    if a >= vh:
        return sign | bh
    dl, dh = a - vl, vh - a
    if dl < dh or (dl == dh and bl % 2 == 0):
        return sign | bl
    return sign | bh


def f32(x):
    """Round a Python float to binary32 (correct: binary64 holds 2p+2 bits)."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def f16_bits_of_float(v):
    """Round a float64 to fp16 bits (ties to even) with integer steps only."""
    import math
    if math.isnan(v):
        return 0x7E00
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if a == 0.0:
        return sign
    if math.isinf(a):
        return sign | 0x7C00
    if a < 2.0 ** -14:
        return sign | round(a * 2.0 ** 24)          # subnormal; 1024 -> min normal
    f, ex = math.frexp(a)                             # a = f * 2^ex, f in [0.5, 1)
    e = ex - 1
    q = round(a * 2.0 ** (10 - e))                    # exact scaling; round() ties to even
    if q == 2048:
        q, e = 1024, e + 1
    if e + 15 >= 31:
        return sign | 0x7C00
    return sign | ((e + 15) << 10) | (q - 1024)


def mul1_bruteforce(state):
    u = (state * 0x83DCD12D) % (1 << 32)
    s = sum((u >> (8 * j)) & 0xFF for j in range(4))
    return nearest_f16_bits(s * f16_value(0x1EEE) + f16_value(0xC2E8))


def bits16(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------------------
# Codebook.
# ---------------------------------------------------------------------------
def test_codebook_all_ones_page_value_every_width():
    for bits_s, state_s, val_s, f16_s in read_golden("codebook_all_ones.txt"):
        k = int(bits_s)
        ones = synth.make_trellis_all_ones(128, 128, k).reshape(8, 8, 8 * k)
        w = o.decode_tiles(ones, k)
        assert np.all(bits16(w) == int(f16_s, 16))
        assert float(w[0, 0, 0, 0]) == float(val_s)
        assert int(state_s, 16) == 0xFFFF


def test_codebook_matches_exact_fma_rounding():
    rng = np.random.default_rng(7)
    states = list(rng.integers(0, 65536, size=1500)) + [0, 1, 0x8000, 0xFFFE, 0xFFFF]
    got = bits16(o.mul1(np.array(states)))
    want = [mul1_bruteforce(int(s)) for s in states]
    assert list(got) == want


def test_codebook_has_no_zero_and_is_gaussian_like():
    w = o.mul1(np.arange(65536)).astype(np.float64)
    assert np.all(w != 0.0)
    assert abs(w.mean()) < 0.01 and abs(w.std() - 1.0) < 0.01


# ---------------------------------------------------------------------------
# Trellis windows and tile layout.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("k", o.BITS_ALLOWED)
def test_windows_match_shift_register_replay(k):
    rng = np.random.default_rng(100 + k)
    for _ in range(3):
        words = rng.integers(0, 2**32, size=8 * k, dtype=np.uint32)
        assert np.array_equal(o.tile_states(words, k), o.tile_states_replay(words, k))


def _words_from_bytes(byte_vals):
    b = bytes(int(v) & 0xFF for v in byte_vals)
    return np.frombuffer(b, dtype=">u4").astype(np.uint32)


def test_hand_tile_8bit():
    # Stream byte j = j: state i is bytes (i-1, i) of the ring.
    words = _words_from_bytes(range(256))
    st = o.tile_states(words, 8)
    for i in range(256):
        assert st[i] == (((i - 1) % 256) << 8) | i
    w = o.decode_tiles(words, 8)                      # [k][n]
    for i in (0, 1, 15, 16, 17, 255):
        k, n = i % 16, i // 16
        assert int(bits16(w[k, n])) == mul1_bruteforce(int(st[i]))


def test_hand_tile_4bit():
    # Nibble j of the stream = j mod 16: state i is nibbles i-3..i (mod 16).
    nib = [j % 16 for j in range(256)]
    byte_vals = [(nib[2 * m] << 4) | nib[2 * m + 1] for m in range(128)]
    st = o.tile_states(_words_from_bytes(byte_vals), 4)
    for i in range(256):
        want = 0
        for d in (3, 2, 1, 0):
            want = (want << 4) | ((i - d) % 16)
        assert st[i] == want
    assert st[3] == 0x0123 and st[0] == 0xDEF0


def test_decode_matrix_tile_placement():
    k = 3
    rng = np.random.default_rng(11)
    i_f, o_f = 256, 128
    tr = rng.integers(0, 2**32, size=i_f * o_f * k // 32, dtype=np.uint32)
    w = o.decode_matrix(tr, i_f, o_f, k)
    per = 8 * k
    for kt in range(i_f // 16):
        for nt in range(o_f // 16):
            words = tr[(kt * (o_f // 16) + nt) * per:(kt * (o_f // 16) + nt + 1) * per]
            st = o.tile_states_replay(words, k)
            for i in (0, 5, 16, 200, 255):
                assert int(bits16(w[16 * kt + i % 16, 16 * nt + i // 16])) == mul1_bruteforce(int(st[i]))
    blk = o.decode_blocks(tr, i_f, o_f, k, [0])
    assert np.array_equal(bits16(blk), bits16(w))


# ---------------------------------------------------------------------------
# Walsh-Hadamard transform.
# ---------------------------------------------------------------------------
def test_fwht_closed_form_and_involution():
    eye = np.eye(128)
    h64 = o.fwht128_f64(eye)          # row j = transform of e_j
    h32 = o.fwht128_f32(eye.astype(np.float32))
    for j in range(128):
        for i in range(128):
            want = -1.0 if bin(i & j).count("1") % 2 else 1.0
            assert h64[j, i] == want and h32[j, i] == want
    v = np.random.default_rng(3).integers(-1000, 1000, size=(5, 128)).astype(np.float64)
    assert np.array_equal(o.fwht128_f64(o.fwht128_f64(v)), 128 * v)


def test_fwht_constant_block_leaves_127_exact_zeros():
    c = -16392192.0
    y = o.fwht128_f64(np.full(128, c))
    assert y[0] == 128 * c and np.all(y[1:] == 0.0)
    y32 = o.fwht128_f32(np.full(128, c, np.float32))
    assert y32[0] == 128 * c and np.all(y32[1:] == 0.0)


def _fwht_f32_loops(v):
    v = [f32(float(t)) for t in v]
    h = 1
    while h < 128:
        for p in range(128):
            if p & h == 0:
                a, b = v[p], v[p + h]
                v[p], v[p + h] = f32(a + b), f32(a - b)
        h *= 2
    return v


def test_fwht_f32_stage_order_against_loops():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((4, 128)).astype(np.float32) * np.float32(3.7)
    got = o.fwht128_f32(v)
    for r in range(4):
        want = np.array(_fwht_f32_loops(v[r]), dtype=np.float32)
        assert np.array_equal(got[r].view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------------------
# rot_in.
# ---------------------------------------------------------------------------
def test_rot_scale_constant_is_nearest_f32():
    s = float(o.f32_from_bits(o.ROT_SCALE_F32_BITS))
    # s^2 * 128 brackets 1 more tightly than either fp32 neighbour's.
    up = float(o.f32_from_bits(o.ROT_SCALE_F32_BITS + 1))
    dn = float(o.f32_from_bits(o.ROT_SCALE_F32_BITS - 1))
    err = lambda t: abs(Fraction(t) ** 2 * 128 - 1)
    assert err(s) < err(up) and err(s) < err(dn)
    # The midpoints to the neighbours lie on opposite sides of 1/sqrt(128).
    mid_up = (Fraction(s) + Fraction(up)) / 2
    mid_dn = (Fraction(s) + Fraction(dn)) / 2
    assert mid_up ** 2 * 128 > 1 > mid_dn ** 2 * 128


def _rot_in_block_loops(x16, s16, mode="ok"):
    """One 128-block by plain loops: fp32 products, fp32 butterflies, fp32
    scale multiply, fp16 rounding by integer steps. `mode` plants one fault:
    "div" divides by fp32 sqrt(128), "f16prod" rounds products to fp16 first,
    "fused" rounds t * scale to fp16 once instead of fp32 then fp16."""
    t = []
    for a, b in zip(x16, s16):
        p = f32(float(a) * float(b))
        if mode == "f16prod":
            p = float(f16_value(f16_bits_of_float(p)))
        t.append(p)
    t = _fwht_f32_loops(t)
    sc = float(o.f32_from_bits(o.ROT_SCALE_F32_BITS))
    if mode == "div":
        t = [f32(v / f32(float(np.sqrt(128.0)))) for v in t]
    elif mode == "fused":
        t = [v * sc for v in t]                       # exact in float64, no fp32 step
    else:
        t = [f32(v * sc) for v in t]
    return [f16_bits_of_float(v) for v in t]


ROT_PIN_ROWS = 1024      # 131,072 roundings: enough for 1-ulp faults to show


def _rot_pin_inputs():
    x = synth.make_x(ROT_PIN_ROWS, 128, 17)
    suh = synth.make_scale(128, 18)
    return x, suh


def test_f16_rounding_helper_against_exact_search():
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(300) * 10.0) + [65519.99, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26,
                                                    1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11]
    for v in vals:
        assert f16_bits_of_float(float(v)) == nearest_f16_bits(Fraction(float(v)))


def test_rot_in_against_plain_loops():
    x, suh = _rot_pin_inputs()
    got = bits16(o.rot_in_f32(x, suh))
    for r in range(ROT_PIN_ROWS):
        assert list(got[r]) == _rot_in_block_loops(x[r], suh)


def test_rot_in_within_float64_bound():
    x = synth.make_x(8, 1024, 21)
    suh = synth.make_scale(1024, 22)
    y16 = o.rot_in_f32(x, suh).astype(np.float64)
    y64 = o.rot_in_f64(x, suh)
    # fp32 steps (depth 8: the product and seven butterflies, then the scale)
    # add at most ~9 * 2^-24 * sum|terms|; the fp16 rounding half an ulp.
    t = np.abs(x.astype(np.float64) * suh.astype(np.float64)).reshape(8, 8, 128).sum(-1)
    bound32 = 9 * 2.0 ** -24 * np.repeat(t, 128, axis=1) / np.sqrt(128.0) * 1.01
    ulp = np.spacing(np.abs(y64).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(y16 - y64) <= bound32 + 0.5 * ulp)


def test_rot_in_input_dtypes():
    x16 = synth.make_x(2, 128, 31)
    suh = synth.make_scale(128, 32)
    a = o.rot_in_f32(x16, suh, "f16")
    b = o.rot_in_f32(x16.astype(np.float32), suh, "f32")
    bf = (x16.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    exact_bf = o.bf16_bits_to_f32(bf)
    assert np.array_equal(bits16(a), bits16(b))
    c = o.rot_in_f32(bf, suh, "bf16")
    assert np.array_equal(bits16(c), bits16(o.rot_in_f32(exact_bf, suh, "f32")))


# ---------------------------------------------------------------------------
# Linear and output rotation.
# ---------------------------------------------------------------------------
def _linear_loops(xr, w, svh):
    rows, i_f = xr.shape
    o_f = w.shape[1]
    out = []
    for r in range(rows):
        acc = [sum(float(xr[r, k]) * float(w[k, n]) for k in range(i_f)) for n in range(o_f)]
        y = []
        for n in range(o_f):
            b, i = divmod(n, 128)
            s = 0.0
            for j in range(128):
                sign = -1.0 if bin(i & j).count("1") % 2 else 1.0
                s += sign * acc[128 * b + j]
            y.append(s / np.sqrt(128.0) * float(svh[n]))
        out.append(y)
    return np.array(out)


@pytest.mark.parametrize("shape", [(1, 128, 128, 4), (3, 128, 128, 2), (2, 256, 128, 6)])
def test_linear_against_bruteforce(shape):
    rows, i_f, o_f, k = shape
    x = synth.make_x(rows, i_f, 41)
    suh = synth.make_scale(i_f, 42)
    svh = synth.make_scale(o_f, 43)
    tr = synth.make_trellis(i_f, o_f, k, 44)
    xr, y = o.project_f64(x, suh, tr, svh, i_f, o_f, k)
    w = o.decode_matrix(tr, i_f, o_f, k)
    want = _linear_loops(xr, w, svh)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-9)


def test_gate4_exact_sums_and_overflow():
    g = {r[0]: r[1] for r in read_golden("gate4_exact.txt")}
    i_f = int(g["in_features"])
    xv = float(g["x_value"])
    wv = float(g["weight"])
    total = Fraction(i_f) * Fraction(xv) * Fraction(wv)
    assert total.denominator == 1 and abs(total) < int(g["sum_magnitude_below"])
    o_f, k = 128, 4
    tr = synth.make_trellis_all_ones(i_f, o_f, k)
    w = o.decode_matrix(tr, i_f, o_f, k)
    xr = np.full((2, i_f), np.float16(xv))
    svh = synth.make_scale(o_f, 51)
    y = o.linear_f64(xr, w, svh)
    acc = xr.astype(np.float64) @ w.astype(np.float64)
    assert np.all(acc == float(total))
    nz = int(g["zero_outputs_per_block"])
    assert np.sum(y[0] == 0.0) == nz and y[0, 0] == float(total) * 128 / np.sqrt(128.0) * float(svh[0])
    y32 = o.epilogue_f32(acc.astype(np.float32), svh)
    assert np.sum(y32[0] == 0.0) == nz
    with np.errstate(over="ignore"):
        y16 = y32.astype(np.float16)
    assert np.isinf(y16[0, 0]) and np.sign(y16[0, 0]) == -np.sign(float(svh[0]))


# ---------------------------------------------------------------------------
# Planted faults: each plausible mistake, made in a copy of an oracle step,
# turns the corresponding pin red.
# ---------------------------------------------------------------------------
def test_planted_codebook_bias_one_ulp_off_is_caught():
    a = float(o.f16_from_bits(o.MUL1_SCALE_BITS))
    b_bad = float(o.f16_from_bits(o.MUL1_BIAS_BITS + 1))
    u = (0xFFFF * o.MUL1_MULTIPLIER) % (1 << 32)
    s = sum((u >> (8 * j)) & 0xFF for j in range(4))
    bad = np.float16(s * a + b_bad)
    assert int(bits16(bad)) != 0xB936


def test_planted_window_one_bit_off_is_caught():
    def states_off(words, k):
        n = 256 * k
        b = o.tile_stream_bits(words)
        i = np.arange(256)[:, None]
        t = np.arange(16)[None, :]
        pos = ((i + 1) * k - 15 + t) % n           # ends one bit late
        win = b[..., pos].astype(np.uint32)
        return (win << (15 - np.arange(16)).astype(np.uint32)).sum(-1)
    words = np.random.default_rng(9).integers(0, 2**32, size=16, dtype=np.uint32)
    assert not np.array_equal(states_off(words, 2), o.tile_states_replay(words, 2))


def _closed_form_ok(fwht):
    h = fwht(np.eye(128))
    for j in range(128):
        for i in range(128):
            if h[j, i] != (-1.0 if bin(i & j).count("1") % 2 else 1.0):
                return False
    return True


def _fwht_variant(v, orientation_flipped=False, reverse_stages=False, dtype=np.float64):
    v = np.array(v, dtype=dtype, copy=True)
    lead = v.shape[:-1]
    hs = [1, 2, 4, 8, 16, 32, 64]
    for h in (hs[::-1] if reverse_stages else hs):
        r = v.reshape(lead + (128 // (2 * h), 2, h))
        a, b = r[..., 0, :], r[..., 1, :]
        lo, hi = (a - b, a + b) if orientation_flipped else (a + b, a - b)
        v = np.stack([lo, hi], axis=-2).reshape(lead + (128,))
    return v


def test_planted_butterfly_orientation_is_caught():
    assert _closed_form_ok(o.fwht128_f64)
    assert _closed_form_ok(_fwht_variant)
    assert not _closed_form_ok(lambda v: _fwht_variant(v, orientation_flipped=True))


def test_planted_stage_order_is_caught_by_fp32_loops():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((4, 128)).astype(np.float32) * np.float32(3.7)
    bad = _fwht_variant(v, reverse_stages=True, dtype=np.float32)
    want = np.array([_fwht_f32_loops(v[r]) for r in range(4)], dtype=np.float32)
    assert not np.array_equal(bad.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("mode", ["div", "f16prod", "fused"])
def test_planted_rot_in_faults_are_caught(mode):
    """Each of the page's three rot_in plants moves some of the pin's outputs."""
    x, suh = _rot_pin_inputs()
    got = bits16(o.rot_in_f32(x, suh))
    moved = sum(sum(a != b for a, b in zip(got[r], _rot_in_block_loops(x[r], suh, mode)))
                for r in range(ROT_PIN_ROWS))
    assert moved > 0


def test_planted_transposed_tile_is_caught():
    k = 4
    tr = synth.make_trellis(128, 128, k, 71)
    w = o.decode_matrix(tr, 128, 128, k)
    t = tr.reshape(8, 8, 8 * k)
    wt = np.swapaxes(o.decode_tiles(t, k), -1, -2)    # n, k swapped inside tiles
    bad = wt.transpose(0, 2, 1, 3).reshape(128, 128)
    assert not np.array_equal(bits16(bad), bits16(w))


def test_decode_rows_and_blocks_agree_with_matrix():
    k = 5
    tr = synth.make_trellis(256, 256, k, 81)
    w = o.decode_matrix(tr, 256, 256, k)
    ks = [0, 17, 255]
    assert np.array_equal(bits16(o.decode_rows(tr, 256, 256, k, ks)), bits16(w[ks]))
    assert np.array_equal(bits16(o.decode_blocks(tr, 256, 256, k, [1])), bits16(w[:, 128:]))


@pytest.mark.parametrize("k", [3, 4, 8])
def test_strips_layout_places_each_word_by_hand_formula(k):
    """Word w of tile (kt, nt) lands at word
    (((b * I/64 + c) * 8 + nt % 8) * 8*bits + p(w)) * 4 + kt % 4 of the
    strips order, with b = nt // 8, c = kt // 4 and p(w) = w at 3 bits,
    p(w) = (w % 2) * 16 + w // 2 at 4 bits (written out below) and
    (w % 4) * 16 + w // 4 at 8 bits."""
    i_f, o_f = 256, 384
    tr = synth.make_trellis(i_f, o_f, k, 91 + k)
    st = o.tiles_to_strips(tr, i_f, o_f, k)
    per = 8 * k
    groups = i_f // 64
    if k == 4:   # even words first, then odd ones
        pos = {w: (w // 2 if w % 2 == 0 else 16 + w // 2) for w in range(per)}
    elif k == 8:
        pos = {w: (w % 4) * 16 + w // 4 for w in range(per)}
    else:
        pos = {w: w for w in range(per)}
    assert sorted(pos.values()) == list(range(per))
    seen = np.zeros(st.size, dtype=bool)
    for kt in range(i_f // 16):
        for nt in range(o_f // 16):
            b, c = nt // 8, kt // 4
            for w in range(per):
                src = (kt * (o_f // 16) + nt) * per + w
                dst = (((b * groups + c) * 8 + nt % 8) * per + pos[w]) * 4 + kt % 4
                assert st[dst] == tr[src]
                seen[dst] = True
    assert seen.all()
    assert np.array_equal(o.strips_to_tiles(st, i_f, o_f, k), tr)


# ------------------------------------------------------------ bf16 output
def test_bf16_rounding_hand_values():
    """bf16 keeps 8 significant bits: at 1.0 the last place is 2^-7."""
    f = lambda v: int(o.bf16_bits_rne(np.float32(v)))
    assert f(1.0) == 0x3F80
    assert f(1.0 + 2.0 ** -8) == 0x3F80           # half a place, kept bit even: stays
    assert f(1.0 + 3 * 2.0 ** -8) == 0x3F82       # half a place, kept bit odd: up to even
    assert f(1.0 + 2.0 ** -8 + 2.0 ** -20) == 0x3F81  # just above half: up
    assert f(-2.5) == 0xC020
    assert f(0.0) == 0x0000 and f(-0.0) == 0x8000
    assert f(np.inf) == 0x7F80 and f(-np.inf) == 0xFF80
    assert f(np.float32(3.4028235e38)) == 0x7F80  # the largest float32 rounds up to infinity
    assert f(np.float32(1e-40)) == int(np.float32(1e-40).view(np.uint32)) >> 16  # subnormal, exact cut
    n = int(o.bf16_bits_rne(np.float32(np.nan)))
    assert (n & 0x7F80) == 0x7F80 and (n & 0x7F) != 0


def test_bf16_rounding_matches_torch():
    """Against torch's float32 -> bfloat16 conversion (nearest, ties to even)
    on random patterns, exact ties and values next to them."""
    torch = pytest.importorskip("torch")
    g = np.random.Generator(np.random.PCG64(1234))
    pat = g.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    ties = (g.integers(0, 2 ** 16, size=20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    pat = np.concatenate([pat, ties, ties + 1, ties - 1])
    v = pat.view(np.float32)
    v = v[~np.isnan(v)]
    want = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.bf16_bits_rne(v), want)


def test_epilogue_f32_within_fp32_bound_of_float64():
    """The fp32-step output epilogue against the float64 one on random sums:
    7 butterfly stages and two multiplies, each rounding at most half an
    fp32 ulp, so |y32 - y64| <= 9 * 2^-24 * 128 * max|acc| * s * |svh| per
    block. A wrong sign, scale, index or dropped term is far outside it."""
    g = np.random.Generator(np.random.PCG64(77))
    acc = g.standard_normal((3, 384)).astype(np.float32) * np.float32(1000.0)
    svh = synth.make_scale(384, 78)
    y32 = o.epilogue_f32(acc, svh).astype(np.float64)
    y64 = o.fwht128_f64(acc.astype(np.float64).reshape(3, 3, 128)).reshape(3, 384) / np.sqrt(128.0)
    y64 = y64 * svh.astype(np.float64)
    amax = np.abs(acc.astype(np.float64)).reshape(3, 3, 128).max(axis=2)          # per block
    bound = 9 * 2.0 ** -24 * 128 * amax / np.sqrt(128.0)
    bound = np.repeat(bound, 128, axis=1) * np.abs(svh.astype(np.float64))
    assert np.all(np.abs(y32 - y64) <= bound)
    # and the bound is tight enough to see a one-element slip
    bad = acc.copy()
    bad[0, 5] += np.float32(1.0)
    assert not np.all(np.abs(o.epilogue_f32(bad, svh).astype(np.float64) - y64) <= bound)

"""CPU oracle for the EXL3-style trellis-quantized projection for decode rows.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import this module. It shares no
code, constant table or helper with the CUDA library; it is written from the
method's description alone and is deliberately plain and slow.

Source: "hip exl3: the input rotation and trellis linear for decode rows,
under the kernel contract" (TensorFold pull request #3314). Section names
below refer to that page.

The method, in four steps:
  1. rot_in: per 128-element block of a row, the fp32 product x * suh, seven
     fp32 butterfly stages of the 128-point Walsh-Hadamard transform, a
     multiply by the fp32 constant 1/sqrt(128), one rounding to fp16
     ("What this changes", first bullet; "Checks on this head", rot_in test).
  2. Decode of 16x16 weight tiles stored as bitshift-trellis streams at
     2, 3, 4, 5, 6 or 8 bits per weight, through the mul1 codebook, with one
     fp16 fma per weight ("What this changes", second bullet).
  3. Each row's K sums (fp32 on the GPU, float64 here).
  4. The output rotation (unscaled butterflies, then the scale, as the page's
     float64 reference does: "Kernel contract", gate 4) and the svh scale.

Readings of points the page leaves open (all recorded in the design notes):
  * mul1 constants: u = (state * 0x83DCD12D) mod 2^32, s = sum of u's four
    bytes, w = fp16_RN(s * a + b) with fp16 a = 0x1EEE and b = 0xC2E8. The
    page fixes only that the all-ones state decodes to -0.6513671875 at every
    width ("Kernel contract", gate 4) and that decoding costs one fp16 fma.
  * Stream bit j of a tile is bit (31 - j mod 32) of word j // 32.
  * The state of weight i is the 16 stream bits ending at bit (i + 1) * bits,
    read circularly (a tail-biting shift register: each weight shifts in
    `bits` new bits).
  * Stream weight i of tile (kt, nt) is W[16*kt + i % 16][16*nt + i // 16]:
    a tile holds each output's 16 input weights consecutively.
  * Tiles are stored k-tile major: tile (kt, nt) is the (kt * O/16 + nt)-th
    run of 8*bits uint32 words.
  * Butterfly stages run h = 1, 2, ..., 64; in each pair (p, p + h) with
    p & h == 0 the lower element becomes a + b and the upper a - b.
  * The output epilogue is: butterflies, times 1/sqrt(128), times svh.

Pins (tests/test_oracle_pins.py) tie each function to something other than
itself: the page's printed codebook value, closed forms of the Hadamard
matrix, a shift-register replay of the windows, hand-derived golden tiles,
brute-force dot products and the page's exact gate-4 integers.
"""

import numpy as np

BITS_ALLOWED = (2, 3, 4, 5, 6, 8)

# mul1 codebook (reading; see module docstring).
MUL1_MULTIPLIER = 0x83DCD12D
MUL1_SCALE_BITS = 0x1EEE   # fp16 0.00676727294921875
MUL1_BIAS_BITS = 0xC2E8    # fp16 -3.453125

# fp32 round-to-nearest of 1/sqrt(128); rot_in multiplies by it ("Checks on
# this head": a division by sqrt(128) is one fp32 ulp off).
ROT_SCALE_F32_BITS = 0x3DB504F3


def f16_from_bits(bits):
    return np.array(bits, dtype=np.uint16).view(np.float16)


def f32_from_bits(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


def bf16_bits_to_f32(bits16):
    """bf16 stored as uint16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits16, dtype=np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Step 2a: the mul1 codebook ("What this changes": mul1, one fp16 fma each).
# ---------------------------------------------------------------------------
def mul1(states):
    """Decode 16-bit trellis states to fp16 weights with the mul1 codebook.

    u = state * M mod 2^32; s = sum of the four bytes of u; the weight is the
    fp16 fma s * a + b rounded once. s * a + b is exact in float64 (s has at
    most 10 bits, a 11 significant bits), so a single float64 -> fp16
    conversion gives the fma's one rounding.
    """
    st = np.asarray(states, dtype=np.uint64)
    u = (st * np.uint64(MUL1_MULTIPLIER)) & np.uint64(0xFFFFFFFF)
    s = (u & np.uint64(0xFF)) + ((u >> np.uint64(8)) & np.uint64(0xFF)) \
        + ((u >> np.uint64(16)) & np.uint64(0xFF)) + (u >> np.uint64(24))
    a = float(f16_from_bits(MUL1_SCALE_BITS))
    b = float(f16_from_bits(MUL1_BIAS_BITS))
    exact = s.astype(np.float64) * a + b
    return exact.astype(np.float16)


# ---------------------------------------------------------------------------
# Step 2b: the bitshift trellis ("What this changes": 16 x 16 tiles at
# 2..8 bits; "Kernel contract", gate 4: all-ones states at every width).
# ---------------------------------------------------------------------------
def tile_stream_bits(words):
    """uint32 words [..., 8*bits] -> stream bits [..., 256*bits], MSB first."""
    w = np.ascontiguousarray(np.asarray(words, dtype=np.uint32))
    be = w.astype(">u4")
    by = be.view(np.uint8).reshape(w.shape[:-1] + (w.shape[-1] * 4,))
    return np.unpackbits(by, axis=-1)


def tile_states(words, bits):
    """16-bit state of each of a tile's 256 weights, read as direct windows.

    State i is the 16 stream bits at positions ((i + 1) * bits - 16 + t) mod
    (256 * bits), t = 0..15, the first bit being the most significant.
    """
    n = 256 * bits
    b = tile_stream_bits(words)
    assert b.shape[-1] == n
    i = np.arange(256)[:, None]
    t = np.arange(16)[None, :]
    pos = ((i + 1) * bits - 16 + t) % n
    win = b[..., pos].astype(np.uint32)
    weight = (np.uint32(1) << (15 - np.arange(16)).astype(np.uint32))
    return (win * weight).sum(axis=-1).astype(np.uint32)


def tile_states_replay(words, bits):
    """The same states from a shift register run around the ring (one tile).

    The register starts at 0 and consumes the stream once to warm up (256 *
    bits >= 16 bits, so it then holds the stream's last 16 bits); on the
    second lap it records its value after shifting in each weight's bits.
    Written independently of tile_states, to pin its windowing.
    """
    b = [int(v) for v in tile_stream_bits(words)]
    assert len(b) == 256 * bits
    groups = []
    for i in range(256):
        g = 0
        for v in b[i * bits:(i + 1) * bits]:
            g = (g << 1) | v
        groups.append(g)
    state = 0
    for g in groups:
        state = ((state << bits) | g) & 0xFFFF
    out = []
    for g in groups:
        state = ((state << bits) | g) & 0xFFFF
        out.append(state)
    return np.array(out, dtype=np.uint32)


def decode_tiles(words, bits):
    """Tiles [..., 8*bits] words -> fp16 [..., 16 (k), 16 (n)] weights.

    Stream weight i sits at input row k = i % 16 and output column n = i // 16.
    """
    w = mul1(tile_states(words, bits))                 # [..., 256], i = 16 n + k
    w = w.reshape(w.shape[:-1] + (16, 16))             # [..., n, k]
    return np.swapaxes(w, -1, -2)                      # [..., k, n]


def check_shape(in_features, out_features, bits):
    assert bits in BITS_ALLOWED
    assert in_features % 128 == 0 and out_features % 128 == 0


def decode_matrix(trellis, in_features, out_features, bits):
    """Whole packed trellis -> dense fp16 W [in_features][out_features]."""
    check_shape(in_features, out_features, bits)
    kt, nt = in_features // 16, out_features // 16
    t = np.asarray(trellis, dtype=np.uint32).reshape(kt, nt, 8 * bits)
    w = decode_tiles(t, bits)                          # [kt, nt, 16k, 16n]
    return np.ascontiguousarray(w.transpose(0, 2, 1, 3)).reshape(in_features, out_features)


def decode_blocks(trellis, in_features, out_features, bits, blocks):
    """Columns of W for the given 128-output blocks: fp16 [in][len(blocks)*128]."""
    check_shape(in_features, out_features, bits)
    kt, nt = in_features // 16, out_features // 16
    t = np.asarray(trellis, dtype=np.uint32).reshape(kt, nt, 8 * bits)
    cols = []
    for b in blocks:
        w = decode_tiles(t[:, 8 * b:8 * b + 8, :], bits)   # [kt, 8, 16k, 16n]
        cols.append(w.transpose(0, 2, 1, 3).reshape(in_features, 128))
    return np.concatenate(cols, axis=1)


# ---------------------------------------------------------------------------
# The 128-point fast Walsh-Hadamard transform (used by steps 1 and 4).
# ---------------------------------------------------------------------------
def _fwht128(v, dtype):
    v = np.array(v, dtype=dtype, copy=True)
    assert v.shape[-1] == 128
    lead = v.shape[:-1]
    h = 1
    while h < 128:
        r = v.reshape(lead + (128 // (2 * h), 2, h))
        a = r[..., 0, :]
        b = r[..., 1, :]
        lo = a + b
        hi = a - b
        v = np.stack([lo, hi], axis=-2).reshape(lead + (128,))
        h *= 2
    return v


def fwht128_f64(v):
    """Unscaled Sylvester butterflies in float64 over the last axis (128)."""
    return _fwht128(v, np.float64)


def fwht128_f32(v):
    """The same butterflies with every add and subtract rounded to fp32."""
    return _fwht128(v, np.float32)


# ---------------------------------------------------------------------------
# Step 1: rot_in ("What this changes", first bullet; the rot_in kernel test).
# ---------------------------------------------------------------------------
def rot_in_input_f32(x, x_dtype):
    """Input rows as float32 (exact for fp16 and bf16, identity for fp32)."""
    if x_dtype == "bf16":
        return bf16_bits_to_f32(x)
    return np.asarray(x).astype(np.float32)


def rot_in_f32(x, suh, x_dtype="f16"):
    """fp16 rows of x rotated by 128: fp32 product, fp32 butterflies, fp32
    scale multiply, one rounding to fp16."""
    x32 = rot_in_input_f32(x, x_dtype)
    rows, n = x32.shape
    assert n % 128 == 0
    t = x32 * np.asarray(suh).astype(np.float32)
    t = fwht128_f32(t.reshape(rows, n // 128, 128)).reshape(rows, n)
    t = t * f32_from_bits(ROT_SCALE_F32_BITS)
    return t.astype(np.float16)


def rot_in_f64(x, suh, x_dtype="f16"):
    """The same rotation in float64 with the exact scale (no rounding)."""
    x64 = rot_in_input_f32(x, x_dtype).astype(np.float64)
    rows, n = x64.shape
    t = x64 * np.asarray(suh).astype(np.float64)
    t = fwht128_f64(t.reshape(rows, n // 128, 128)).reshape(rows, n)
    return t / np.sqrt(128.0)


# ---------------------------------------------------------------------------
# Steps 3 and 4: the linear and its output rotation ("Kernel contract":
# the float64 reference sums each output's K terms, then rotates with
# unscaled butterflies, then scales).
# ---------------------------------------------------------------------------
def linear_f64(xr, w, svh):
    """y = svh * (1/sqrt(128)) * FWHT_128(xr @ W), all in float64.

    xr: fp16 [rows][in] (the rotated rows the GPU consumes), w: fp16
    [in][out], svh: fp16 [out]. Returns float64 [rows][out].
    """
    acc = np.asarray(xr).astype(np.float64) @ np.asarray(w).astype(np.float64)
    rows, n = acc.shape
    y = fwht128_f64(acc.reshape(rows, n // 128, 128)).reshape(rows, n)
    y = y * (1.0 / np.sqrt(128.0))
    return y * np.asarray(svh).astype(np.float64)


def epilogue_f32(acc32, svh):
    """The output rotation with fp32 steps: butterflies, * fp32 1/sqrt(128),
    * fp32 svh. Used where the K sums are exact (identity rows, gate 4)."""
    a = np.asarray(acc32, dtype=np.float32)
    rows, n = a.shape
    y = fwht128_f32(a.reshape(rows, n // 128, 128)).reshape(rows, n)
    y = y * f32_from_bits(ROT_SCALE_F32_BITS)
    return y * np.asarray(svh).astype(np.float32)


def bf16_bits_rne(y32):
    """float32 values -> bf16 bit patterns (uint16), rounded once to nearest
    with ties to even ("Checks on this head": the linear at 4 bits with bf16
    out). bf16 keeps the top 16 bits of the float32 pattern; the dropped low
    16 bits round the kept part up when they exceed half of its last place,
    or equal half and the kept last bit is odd. A carry out of the fraction
    moves to the next exponent, so the largest values round to infinity.
    NaN stays NaN (quiet, sign kept)."""
    y = np.asarray(y32, dtype=np.float32)
    b = y.view(np.uint32).astype(np.uint64)
    kept, dropped = b >> 16, b & 0xFFFF
    up = (dropped > 0x8000) | ((dropped == 0x8000) & ((kept & 1) == 1))
    out = kept + up.astype(np.uint64)
    out = np.where(np.isnan(y), kept | 0x40, out)
    return out.astype(np.uint16)


def project_f64(x, suh, trellis, svh, in_features, out_features, bits, x_dtype="f16"):
    """The whole path: rot_in (fp32 steps, fp16 out), decode, float64 linear."""
    xr = rot_in_f32(x, suh, x_dtype)
    w = decode_matrix(trellis, in_features, out_features, bits)
    return xr, linear_f64(xr, w, svh)


def decode_rows(trellis, in_features, out_features, bits, ks):
    """Rows W[k, :] for the given input indices: fp16 [len(ks)][out_features]."""
    check_shape(in_features, out_features, bits)
    kt, nt = in_features // 16, out_features // 16
    t = np.asarray(trellis, dtype=np.uint32).reshape(kt, nt, 8 * bits)
    out = []
    for k in ks:
        w = decode_tiles(t[k // 16], bits)               # [nt, 16k, 16n]
        out.append(w[:, k % 16, :].reshape(out_features))
    return np.stack(out)


# ---------------------------------------------------------------------------
# The second storage order of the same tiles ("Checks on this head": the
# decode test runs on the checkpoint's tile layout and on the strips layout).
# Reading (the page does not specify it): a strip is one block of 128
# outputs, stored whole; inside it, groups of four k-tiles follow in input
# order, and a group stores its 8 n-tiles one after another with the words of
# its four k-tiles interleaved: word w of k-tiles 4c, 4c+1, 4c+2, 4c+3 are
# four consecutive words (a quad). Within an n-tile of a group the quads are
# dealt out by w mod s, s = bits / 2 at 4 and 8 bits and 1 otherwise: quad w
# is the (w mod s) * (8 bits / s) + w // s -th. Every word of the tiles
# appears once.
# ---------------------------------------------------------------------------
def strips_quad_positions(bits):
    """Position of quad w inside an n-tile of a group, for w = 0 .. 8 bits - 1."""
    s = bits // 2 if bits in (4, 8) else 1
    per = 8 * bits // s
    return [(w % s) * per + w // s for w in range(8 * bits)]


def tiles_to_strips(trellis, in_features, out_features, bits):
    """k-tile-major packed tiles -> strips order (same words, other order)."""
    check_shape(in_features, out_features, bits)
    kt, nt = in_features // 16, out_features // 16
    t = np.asarray(trellis, dtype=np.uint32).reshape(kt // 4, 4, nt // 8, 8, 8 * bits)
    # [group][kt%4][block][nt%8][word] -> [block][group][nt%8][word][kt%4]
    g = t.transpose(2, 0, 3, 4, 1)
    out = np.empty_like(g)
    out[:, :, :, strips_quad_positions(bits), :] = g
    return np.ascontiguousarray(out).reshape(-1)


def strips_to_tiles(strips, in_features, out_features, bits):
    check_shape(in_features, out_features, bits)
    kt, nt = in_features // 16, out_features // 16
    s = np.asarray(strips, dtype=np.uint32).reshape(nt // 8, kt // 4, 8, 8 * bits, 4)
    s = s[:, :, :, strips_quad_positions(bits), :]   # back to word order
    # [block][group][nt%8][word][kt%4] -> [group][kt%4][block][nt%8][word]
    return np.ascontiguousarray(s.transpose(1, 4, 0, 2, 3)).reshape(-1)

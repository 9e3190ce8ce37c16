"""Seeded synthetic inputs for the trellis-quantized projection.

This module only draws random numbers and builds trivially structured arrays
(an identity, a constant, all-ones words). It holds none of the method's
arithmetic, so both the CUDA path's tests and the float64 oracle can take
their inputs from it without sharing any of the computation.

Distributions follow the workloads of "hip exl3: the input rotation and
trellis linear for decode rows" (section "What this changes"): activation
rows x ~ N(0, 1) in fp16, per-channel scales suh / svh drawn as a random
sign times U[0.5, 1.5] in fp16, and the packed trellis words uniformly
random (every tile's 256*bits-bit stream is a uniform random bit string).
"""

import numpy as np

# Seeds per workload: x = 1000 + c, suh = 2000 + c, svh = 3000 + c,
# trellis = 4000 + c + bits, where c identifies the workload.
SEED_X, SEED_SUH, SEED_SVH, SEED_TRELLIS = 1000, 2000, 3000, 4000

# Shapes of the three projections the page serves (out x in).
SHAPES = {
    "wk": (512, 128),          # indexer's wk: 512 -> 128
    "wkv": (6144, 25600),      # Engram's wkv: 6144 -> 25,600
    "head": (5120, 129280),    # LM head: 5120 -> 129,280
}


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def make_x(rows, in_features, seed, dtype=np.float16):
    """Activation rows, N(0, 1), [rows][in_features], row-major."""
    v = _rng(seed).standard_normal((rows, in_features))
    return v.astype(dtype)


def make_scale(n, seed):
    """suh / svh: random sign times U[0.5, 1.5], fp16, length n."""
    g = _rng(seed)
    sign = np.where(g.integers(0, 2, size=n) == 1, 1.0, -1.0)
    mag = g.uniform(0.5, 1.5, size=n)
    return (sign * mag).astype(np.float16)


def trellis_words(in_features, out_features, bits):
    """Number of uint32 words the packed trellis of a projection occupies."""
    return in_features * out_features * bits // 32


def make_trellis(in_features, out_features, bits, seed):
    """Uniformly random packed trellis words (uint32)."""
    n = trellis_words(in_features, out_features, bits)
    return _rng(seed).integers(0, 2**32, size=n, dtype=np.uint32)


def make_trellis_all_ones(in_features, out_features, bits):
    """Every stream bit set: every 16-bit state is 0xFFFF."""
    return np.full(trellis_words(in_features, out_features, bits), 0xFFFFFFFF, np.uint32)


def make_identity_rows(rows, in_features, ks, negative_zero=False):
    """Rows of the identity: row r is e_{ks[r]} (value 1.0), +0 (or -0) elsewhere."""
    fill = np.float16(-0.0) if negative_zero else np.float16(0.0)
    x = np.full((rows, in_features), fill, np.float16)
    for r, k in enumerate(ks):
        x[r, k] = np.float16(1.0)
    return x


def identity_ks(rows, in_features):
    """Distinct input indices for an identity run: k_r = (r*(I/8) + 17*r) mod I."""
    ks = [(r * (in_features // 8) + 17 * r) % in_features for r in range(rows)]
    assert len(set(ks)) == rows
    return ks


def random_windows(total_rows, count, seed, lo=2, hi=24):
    """(first_row, length) windows of lo..hi rows inside [0, total_rows)."""
    g = _rng(seed)
    out = []
    for _ in range(count):
        n = int(g.integers(lo, hi + 1))
        first = int(g.integers(0, total_rows - n + 1))
        out.append((first, n))
    return out

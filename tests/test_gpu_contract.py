"""GPU checks after the page's kernel contract: the launch the benchmark
times, checked element by element against the oracle at its own shape and
at every output block its work split cuts between CTAs; the contract's
planted controls (the real kernels launched wrongly from the host must go
red); rows past the batch left untouched; the contract's shape list at every
width with five byte-identical runs; non-finite inputs in every input dtype;
calls back to back on one stream and one workspace; a decode step replayed
from a CUDA graph; and the codebook at every one of the 65,536 trellis
states.

Page: "hip exl3: the input rotation and trellis linear for decode rows"
(TensorFold pull request #3314), sections "Checks on this head" and "Kernel
contract".
"""

import numpy as np
import pytest

from oracle import exl3 as o
from trellis_quantized_linear_rot_gb300 import synth
from helpers import assert_close_f32, bits16, cut_blocks, dev, dev_bf16, host, rel_err_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import trellis_quantized_linear_rot_gb300 as tf  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tf.lib()
    yield
    tf.tf_device_error()


def num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def inputs(rows, i_f, o_f, bits, c):
    x = synth.make_x(rows, i_f, synth.SEED_X + c)
    suh = synth.make_scale(i_f, synth.SEED_SUH + c)
    svh = synth.make_scale(o_f, synth.SEED_SVH + c)
    tr = synth.make_trellis(i_f, o_f, bits, synth.SEED_TRELLIS + c + bits)
    return x, suh, svh, tr


def block_cols(blocks):
    return np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])


# ------------------------------------------------- the benchmark's own launch
@pytest.fixture(scope="module")
def head():
    """The benchmark's workload: LM head 5120 -> 129,280 at 4 bits, fp32
    logits, the weights in both orders (the k-tile order the benchmark times
    by default, and the strips order of its --layout strips); the oracle's
    weights of the first, second and last blocks and of every block the
    launch cuts between CTAs."""
    i_f, o_f, bits = 5120, 129280, 4
    x, suh, svh, tr = inputs(16, i_f, o_f, bits, c=2)
    blocks = sorted({0, 1, o_f // 128 - 1} | set(cut_blocks(num_sms(), i_f, o_f, bits)))
    w = o.decode_blocks(tr, i_f, o_f, bits, blocks)
    tiles_t = dev(tr)
    strips_t = tf.tf_trellis_to_strips(tiles_t, i_f, o_f, bits)
    return dict(i_f=i_f, o_f=o_f, bits=bits, x=x, suh=suh, svh=svh, tiles=tiles_t, strips=strips_t,
                blocks=blocks, w=w)


@pytest.mark.parametrize("layout", ["tiles", "strips"])
@pytest.mark.parametrize("rows", [1, 8, 16])
def test_benchmark_launch_matches_oracle_at_every_cut_block(head, rows, layout):
    """rot_in then the linear exactly as the benchmark launches them (same
    shape, weight order, output dtype and CTA count), compared with the
    float64 oracle element by element on the blocks whose sums are split
    between CTAs (the cross-CTA partial-sum path), and the first and last
    blocks; every output is finite."""
    h = head
    assert len(h["blocks"]) > 100
    xr_t = tf.tf_rot_in(dev(h["x"][:rows]), dev(h["suh"]))
    linear = tf.tf_trellis_linear if layout == "tiles" else tf.tf_trellis_linear_strips
    y = host(linear(xr_t, h[layout], dev(h["svh"]), h["bits"], h["o_f"], out_dtype=torch.float32))
    tf.tf_device_error()
    assert np.all(np.isfinite(y))
    cols = block_cols(h["blocks"])
    ref = o.linear_f64(host(xr_t), h["w"], h["svh"][cols])
    assert_close_f32(y[:, cols], ref)


# ---------------------------------------------------------- planted controls
def test_planted_control_rot_in_reading_the_next_blocks_suh_goes_red():
    """"Kernel contract", planted controls: rot_in launched with suh one
    128-block late (a suh buffer with 128 extra entries, passed 128 entries
    in) must fail the bit-exact check that the correct launch passes."""
    rows, i_f = 64, 512
    x = synth.make_x(rows, i_f, 7001)
    suh_ext = synth.make_scale(i_f + 128, 7002)
    want = o.rot_in_f32(x, suh_ext[:i_f])
    suh_t = dev(suh_ext)
    good = host(tf.tf_rot_in(dev(x), suh_t[:i_f]))
    assert np.array_equal(bits16(good), bits16(want))
    planted = host(tf.tf_rot_in(dev(x), suh_t[128:]))
    assert not np.array_equal(bits16(planted), bits16(want)), "the planted control stayed green"


def test_planted_control_linear_reading_rows_one_late_goes_red():
    """"Kernel contract", planted controls: the linear launched on its input
    rows one row late (an xr buffer with one extra row, passed one row in)
    must fail the oracle bound that the correct launch meets, by a wide
    margin."""
    rows, i_f, o_f, bits = 16, 128, 512, 4
    x, suh, svh, tr = inputs(rows + 1, i_f, o_f, bits, c=71)
    xr = o.rot_in_f32(x, suh)
    ref = o.linear_f64(xr[:rows], o.decode_matrix(tr, i_f, o_f, bits), svh)
    xr_t, tr_t, svh_t = dev(xr), dev(tr), dev(svh)
    good = host(tf.tf_trellis_linear(xr_t[:rows], tr_t, svh_t, bits, o_f, out_dtype=torch.float32))
    assert_close_f32(good, ref)
    planted = host(tf.tf_trellis_linear(xr_t[1:], tr_t, svh_t, bits, o_f, out_dtype=torch.float32))
    err = rel_err_rows(planted, ref)
    assert err.max() > 100 * 1e-4, "the planted control stayed green (%.2e)" % err.max()


# ------------------------------------------------------------------ canaries
@pytest.mark.parametrize("rows", [1, 8, 15, 17])
def test_rows_past_the_batch_are_untouched(rows):
    """y allocated with two extra rows holding a sentinel: the call writes
    its rows (matching the oracle) and leaves the two sentinel rows as they
    were."""
    i_f, o_f, bits = 1024, 2048, 4
    x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=80 + rows)
    xr = o.rot_in_f32(x, suh)
    ref = o.linear_f64(xr, o.decode_matrix(tr, i_f, o_f, bits), svh)
    sentinel = np.float32(-1.25e30)
    y_t = torch.full((rows + 2, o_f), float(sentinel), dtype=torch.float32, device="cuda")
    tf.tf_trellis_linear(dev(xr), dev(tr), dev(svh), bits, o_f, y=y_t[:rows])
    tf.tf_device_error()
    y = host(y_t)
    assert np.all(y[rows:] == sentinel)
    assert_close_f32(y[:rows], ref)


# ----------------------------------------------------- contract shape list
CONTRACT_SHAPES = [
    # (in, out, rows): the plan's edge (8192 x 1024 at 4 and 16 rows) and the
    # shape below it (8064 x 1024), gate 4's Engram K at one row of one
    # column block (128 x 6144), the row edges at K and N of 128 and 256.
    (1024, 8192, (4, 16)),
    (1024, 8064, (4,)),
    (6144, 128, (1,)),
    (128, 128, (1, 15, 16, 17, 64)),
    (256, 256, (1, 15, 16, 17, 64)),
]


@pytest.mark.parametrize("bits", o.BITS_ALLOWED)
@pytest.mark.parametrize("i_f,o_f,rows_list", CONTRACT_SHAPES)
def test_contract_shapes_match_oracle_and_repeat_byte_identical(bits, i_f, o_f, rows_list):
    """"Kernel contract": the registration's shapes at every width, fp32
    out, each element within the oracle bound; five runs of each are
    byte-identical."""
    x, suh, svh, tr = inputs(max(rows_list), i_f, o_f, bits, c=90)
    w = o.decode_matrix(tr, i_f, o_f, bits)
    xr_all = o.rot_in_f32(x, suh)
    tr_t, svh_t = dev(tr), dev(svh)
    for rows in rows_list:
        xr_t = dev(xr_all[:rows])
        runs = [host(tf.tf_trellis_linear(xr_t, tr_t, svh_t, bits, o_f, out_dtype=torch.float32)).tobytes()
                for _ in range(5)]
        tf.tf_device_error()
        assert all(r == runs[0] for r in runs), "%d rows: runs differ" % rows
        y = np.frombuffer(runs[0], dtype=np.float32).reshape(rows, o_f)
        assert_close_f32(y, o.linear_f64(xr_all[:rows], w, svh))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_rot_in_non_finite_classes_every_input_dtype(dtype):
    """"Kernel contract": rot_in's non-finite outputs match float64's classes
    (NaN, +inf, -inf) from fp16, bf16 and fp32 rows, and every block without
    a non-finite input stays finite."""
    rows, i_f = 3, 384
    x32 = synth.make_x(rows, i_f, 9100, dtype=np.float32)
    x32[0, 5] = np.inf
    x32[1, 200] = np.nan
    x32[2, 300] = -np.inf
    suh = synth.make_scale(i_f, 9101)
    if dtype == "f16":
        x_np = x32.astype(np.float16)
        x_t = dev(x_np)
    elif dtype == "f32":
        x_np = x32
        x_t = dev(x_np)
    else:
        x_np = (x32.view(np.uint32) >> 16).astype(np.uint16)
        x_t = dev_bf16(x_np)
    got = host(tf.tf_rot_in(x_t, dev(suh))).astype(np.float64)
    want = o.rot_in_f64(x_np, suh, dtype)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(np.isposinf(got), np.isposinf(want))
    assert np.array_equal(np.isneginf(got), np.isneginf(want))
    assert np.all(np.isfinite(got[0, 128:])) and np.all(np.isfinite(got[1, :128]))
    assert np.all(np.isfinite(got[2, :256]))


# --------------------------------------------------- calls back to back
def test_back_to_back_calls_on_one_stream_and_workspace():
    """Different shapes, row counts and output dtypes issued back to back on
    one stream with nothing in between (each linear may start while the
    previous kernel finishes, and all share the library's workspace): every
    result matches the oracle."""
    cases = [(2048, 8192, 4, 16, torch.float32), (1024, 4096, 6, 3, torch.float32),
             (512, 1024, 2, 40, torch.float32), (2048, 8192, 4, 1, torch.float32)]
    prepared, outs = [], []
    for k, (i_f, o_f, bits, rows, dt) in enumerate(cases):
        x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=120 + k)
        prepared.append((x, suh, svh, tr, dev(x), dev(suh), dev(svh), dev(tr)))
    torch.cuda.synchronize()
    for (i_f, o_f, bits, rows, dt), p in zip(cases, prepared):
        xr_t = tf.tf_rot_in(p[4], p[5])
        outs.append((xr_t, tf.tf_trellis_linear(xr_t, p[7], p[6], bits, o_f, out_dtype=dt)))
    tf.tf_device_error()
    for (i_f, o_f, bits, rows, dt), p, (xr_t, y_t) in zip(cases, prepared, outs):
        x, suh, svh, tr = p[:4]
        xr = host(xr_t)
        assert np.array_equal(bits16(xr), bits16(o.rot_in_f32(x, suh)))
        assert_close_f32(host(y_t), o.linear_f64(xr, o.decode_matrix(tr, i_f, o_f, bits), svh))


# ------------------------------------------------- replay in a CUDA graph
def test_rot_in_and_linear_replay_in_a_cuda_graph_bit_identical():
    """A decode step captured once in a CUDA graph (rot_in and the linear for
    three layers of different shapes, widths and row counts, all on the
    library's one workspace) and replayed: every replay gives the eager
    results bit for bit, and the eager results match the oracle. The launches
    hold no allocation and no synchronisation once the workspace exists."""
    cases = [(512, 128, 4, 1), (6144, 1024, 6, 4), (2048, 8192, 3, 16)]
    prepared = []
    for k, (i_f, o_f, bits, rows) in enumerate(cases):
        x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=140 + k)
        prepared.append((x, suh, svh, tr, dev(x), dev(suh), dev(svh), dev(tr)))
    eager = []
    for (i_f, o_f, bits, rows), p in zip(cases, prepared):
        xr_t = tf.tf_rot_in(p[4], p[5])
        eager.append(host(tf.tf_trellis_linear(xr_t, p[7], p[6], bits, o_f)))
    torch.cuda.synchronize()
    tf.tf_device_error()
    # outputs and intermediates the graph writes into
    xrs = [torch.empty((rows, i_f), dtype=torch.float16, device="cuda") for (i_f, o_f, bits, rows) in cases]
    ys = [torch.empty((rows, o_f), dtype=torch.float32, device="cuda") for (i_f, o_f, bits, rows) in cases]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for (i_f, o_f, bits, rows), p, xr_t, y_t in zip(cases, prepared, xrs, ys):
            tf.tf_rot_in(p[4], p[5], xr=xr_t)
            tf.tf_trellis_linear(xr_t, p[7], p[6], bits, o_f, y=y_t)
    for _ in range(3):
        for y_t in ys:
            y_t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        tf.tf_device_error()
        for want, y_t in zip(eager, ys):
            assert np.array_equal(host(y_t).view(np.uint32), want.view(np.uint32))
    for (i_f, o_f, bits, rows), p, want in zip(cases, prepared, eager):
        x, suh, svh, tr = p[:4]
        xr = o.rot_in_f32(x, suh)
        assert_close_f32(want, o.linear_f64(xr, o.decode_matrix(tr, i_f, o_f, bits), svh))


# ------------------------------------------------- every codebook state
def all_states_trellis():
    """An 8-bit trellis of 512 tiles (in = 512, out = 256) whose windows hold
    every 16-bit state: at 8 bits the state of weight i is stream bytes
    (i - 1, i), so a tile whose bytes alternate a, x0, a, x1, ..., a, x127
    holds the states (a, x_m) and (x_m, a); two tiles per value of a (x over
    0..127 and over 128..255) cover all 65,536."""
    i_f, o_f = 512, 256
    n_tiles = (i_f // 16) * (o_f // 16)
    tiles = np.zeros((n_tiles, 256), dtype=np.uint8)
    for tix in range(n_tiles):
        a, half = tix // 2, tix % 2
        tiles[tix, 0::2] = a
        tiles[tix, 1::2] = np.arange(128) + 128 * half
    # Stream byte 4j is the most significant byte of word j.
    words = tiles.reshape(n_tiles, 64, 4).astype(np.uint32)
    words = (words[:, :, 0] << 24) | (words[:, :, 1] << 16) | (words[:, :, 2] << 8) | words[:, :, 3]
    return words.reshape(-1).astype(np.uint32), i_f, o_f


def test_decode_covers_every_codebook_state_bit_for_bit():
    """tf_trellis_decode and the linear's own decode (identity rows through
    the output rotation, passes of 128 rows) against the oracle's mul1 at
    all 65,536 states, bit for bit."""
    tr, i_f, o_f = all_states_trellis()
    bits = 8
    words = tr.reshape(-1, 8 * bits)
    states = np.concatenate([o.tile_states(wd, bits) for wd in words])
    assert np.unique(states).size == 65536
    w_ref = o.decode_matrix(tr, i_f, o_f, bits)
    w_gpu = host(tf.tf_trellis_decode(dev(tr), i_f, o_f, bits))
    assert np.array_equal(bits16(w_gpu), bits16(w_ref))
    assert np.array_equal(np.sort(bits16(w_ref).reshape(-1)), np.sort(bits16(o.mul1(states))))
    # Through the linear: row k of the identity picks weight row k.
    svh = synth.make_scale(o_f, 9200)
    ks = list(range(i_f))
    xr = synth.make_identity_rows(i_f, i_f, ks)
    y = host(tf.tf_trellis_linear(dev(xr), dev(tr), dev(svh), bits, o_f, out_dtype=torch.float32))
    tf.tf_device_error()
    want = o.epilogue_f32(w_ref.astype(np.float32), svh)
    assert np.array_equal(y.view(np.uint32), want.view(np.uint32))

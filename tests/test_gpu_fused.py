"""GPU checks of tf_rot_in_linear, the rotation and the linear in one launch
per pass: its xr and y are the bits of tf_rot_in followed by
tf_trellis_linear at every width, input and output dtype and row count
(passes of 128 rows included); calls of different shapes back to back on one
stream; a CUDA graph of fused calls replayed; and one case against the
float64 oracle directly.

Page: "hip exl3: the input rotation and trellis linear for decode rows"
(TensorFold pull request #3314), section "What this changes" (rot_in, then
the linear, for each projection).
"""

import numpy as np
import pytest

from oracle import exl3 as o
from trellis_quantized_linear_rot_gb300 import synth
from helpers import assert_close_f32, dev, host

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


DT = {"f16": torch.float16, "f32": torch.float32, "bf16": torch.bfloat16}


def make(rows, i_f, o_f, bits, c, x_dtype="f16"):
    x = synth.make_x(rows, i_f, synth.SEED_X + c)
    suh = synth.make_scale(i_f, synth.SEED_SUH + c)
    svh = synth.make_scale(o_f, synth.SEED_SVH + c)
    tr = synth.make_trellis(i_f, o_f, bits, synth.SEED_TRELLIS + c + bits)
    x_t = dev(x.astype(np.float32)).to(DT[x_dtype]) if x_dtype != "f16" else dev(x)
    return x, suh, svh, tr, x_t, dev(suh), dev(svh), dev(tr)


def bits_of(t):
    return host(t).view(np.uint16 if t.element_size() == 2 else np.uint32)


def separate(x_t, suh_t, tr_t, svh_t, bits, o_f, out_dtype):
    xr = tf.tf_rot_in(x_t, suh_t)
    return xr, tf.tf_trellis_linear(xr, tr_t, svh_t, bits, o_f, out_dtype=out_dtype)


CASES = [
    # (in, out, bits, rows, x dtype, out dtype)
    (5120, 129280, 4, 1, "f16", "f32"),
    (5120, 129280, 4, 8, "f16", "f32"),
    (5120, 129280, 4, 16, "f16", "f32"),
    (6144, 25600, 4, 1, "f16", "f16"),
    (6144, 25600, 4, 4, "f16", "f16"),
    (6144, 25600, 4, 16, "f16", "f16"),
    (512, 128, 4, 1, "f16", "f16"),
    (2048, 4096, 2, 8, "f16", "f16"),
    (2048, 4096, 3, 8, "bf16", "f16"),
    (2048, 4096, 5, 8, "f32", "f16"),
    (2048, 4096, 6, 8, "f16", "bf16"),
    (2048, 4096, 8, 8, "f16", "f32"),
    (1024, 2048, 4, 17, "f16", "f32"),
    (1024, 2048, 4, 64, "f16", "f32"),
    (1024, 1024, 6, 130, "bf16", "f32"),  # two passes: 128 rows, then 2
    (128, 6144, 4, 3, "f32", "bf16"),
]


@pytest.mark.parametrize("i_f,o_f,bits,rows,xdt,odt", CASES)
def test_fused_is_rot_in_then_linear_bit_for_bit(i_f, o_f, bits, rows, xdt, odt):
    x, suh, svh, tr, x_t, suh_t, svh_t, tr_t = make(rows, i_f, o_f, bits, c=300 + bits, x_dtype=xdt)
    xr_s, y_s = separate(x_t, suh_t, tr_t, svh_t, bits, o_f, DT[odt])
    xr_f = torch.full_like(xr_s, float("nan"))
    y_f = torch.full_like(y_s, float("nan"))
    tf.tf_rot_in_linear(x_t, suh_t, tr_t, svh_t, bits, o_f, xr=xr_f, y=y_f)
    torch.cuda.synchronize()
    tf.tf_device_error()
    assert np.array_equal(bits_of(xr_f), bits_of(xr_s))
    assert np.array_equal(bits_of(y_f), bits_of(y_s))


@pytest.mark.parametrize("i_f,o_f,bits,rows", [(5120, 129280, 4, 1), (5120, 129280, 4, 16), (2048, 4096, 6, 24),
                                                (1024, 2048, 3, 130)])
def test_fused_strips_is_rot_in_then_strips_linear_bit_for_bit(i_f, o_f, bits, rows):
    """tf_rot_in_linear_strips: the bits of tf_rot_in then tf_trellis_linear_strips, and of the fused
    call on the same weights in the k-tile order."""
    x, suh, svh, tr, x_t, suh_t, svh_t, tr_t = make(rows, i_f, o_f, bits, c=350 + bits)
    strips_t = tf.tf_trellis_to_strips(tr_t, i_f, o_f, bits)
    xr_s = tf.tf_rot_in(x_t, suh_t)
    y_s = tf.tf_trellis_linear_strips(xr_s, strips_t, svh_t, bits, o_f, out_dtype=torch.float32)
    xr_f, y_f = tf.tf_rot_in_linear(x_t, suh_t, strips_t, svh_t, bits, o_f, out_dtype=torch.float32, strips=True)
    _, y_t = tf.tf_rot_in_linear(x_t, suh_t, tr_t, svh_t, bits, o_f, out_dtype=torch.float32)
    torch.cuda.synchronize()
    tf.tf_device_error()
    assert np.array_equal(bits_of(xr_f), bits_of(xr_s))
    assert np.array_equal(bits_of(y_f), bits_of(y_s))
    assert np.array_equal(bits_of(y_f), bits_of(y_t))


def test_fused_matches_the_oracle():
    """The fused call against the float64 oracle directly (xr bit-exact with
    the oracle's fp32 rotation, y within the 1e-4 bound), at a shape whose
    work is cut between CTAs."""
    rows, i_f, o_f, bits = 5, 1024, 4096, 4
    x, suh, svh, tr, x_t, suh_t, svh_t, tr_t = make(rows, i_f, o_f, bits, c=321)
    xr_t, y_t = tf.tf_rot_in_linear(x_t, suh_t, tr_t, svh_t, bits, o_f, out_dtype=torch.float32)
    tf.tf_device_error()
    want_xr = o.rot_in_f32(x, suh)
    assert np.array_equal(host(xr_t).view(np.uint16), np.asarray(want_xr, np.float16).view(np.uint16))
    assert_close_f32(host(y_t), o.linear_f64(want_xr, o.decode_matrix(tr, i_f, o_f, bits), svh))


def test_fused_calls_of_different_shapes_back_to_back():
    """Fused and separate calls interleaved on one stream with no
    synchronisation between them (each launch overlaps the one before it):
    every output equals the same call made alone."""
    shapes = [(5120, 8192, 4, 16), (512, 128, 4, 1), (6144, 2048, 6, 4), (2048, 4096, 2, 9), (5120, 8192, 4, 1)]
    data = [make(r, i, o_, b, c=330 + k) for k, (i, o_, b, r) in enumerate(shapes)]
    alone = []
    for (i_f, o_f, bits, rows), d in zip(shapes, data):
        xr, y = separate(d[4], d[5], d[7], d[6], bits, o_f, torch.float32)
        torch.cuda.synchronize()
        alone.append((bits_of(xr), bits_of(y)))
    outs = []
    for k, ((i_f, o_f, bits, rows), d) in enumerate(zip(shapes, data)):
        if k % 2 == 0:
            outs.append(tf.tf_rot_in_linear(d[4], d[5], d[7], d[6], bits, o_f, out_dtype=torch.float32))
        else:
            outs.append(separate(d[4], d[5], d[7], d[6], bits, o_f, torch.float32))
    torch.cuda.synchronize()
    tf.tf_device_error()
    for (xr, y), (want_xr, want_y) in zip(outs, alone):
        assert np.array_equal(bits_of(xr), want_xr)
        assert np.array_equal(bits_of(y), want_y)


def test_fused_calls_replay_in_a_cuda_graph_bit_identical():
    """Fused calls of three shapes captured in one CUDA graph and replayed
    three times: every replay gives the eager results bit for bit (the
    launch's hand-over counts return to zero after each launch)."""
    cases = [(512, 128, 4, 1), (6144, 1024, 6, 4), (2048, 8192, 3, 16)]
    data = [make(r, i, o_, b, c=340 + k) for k, (i, o_, b, r) in enumerate(cases)]
    eager = []
    for (i_f, o_f, bits, rows), d in zip(cases, data):
        xr, y = tf.tf_rot_in_linear(d[4], d[5], d[7], d[6], bits, o_f, out_dtype=torch.float32)
        torch.cuda.synchronize()
        eager.append((bits_of(xr), bits_of(y)))
    tf.tf_device_error()
    xrs = [torch.empty((rows, i_f), dtype=torch.float16, device="cuda") for (i_f, o_f, bits, rows) in cases]
    ys = [torch.empty((rows, o_f), dtype=torch.float32, device="cuda") for (i_f, o_f, bits, rows) in cases]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for (i_f, o_f, bits, rows), d, xr_t, y_t in zip(cases, data, xrs, ys):
            tf.tf_rot_in_linear(d[4], d[5], d[7], d[6], bits, o_f, xr=xr_t, y=y_t)
    for _ in range(3):
        for xr_t, y_t in zip(xrs, ys):
            xr_t.fill_(float("nan"))
            y_t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        tf.tf_device_error()
        for (want_xr, want_y), xr_t, y_t in zip(eager, xrs, ys):
            assert np.array_equal(bits_of(xr_t), want_xr)
            assert np.array_equal(bits_of(y_t), want_y)

"""The allocation-free entry point, tf_trellis_linear_noalloc, against the
regular one, through the C ABI on the GPU.

It exists for callers that cannot let the library call cudaMalloc: for
example a serving process whose caching allocator already holds the device
memory it plans around, or code that must not risk the implicit device
synchronisation an allocation can cause. Its scratch lives in a fixed device
array instead. This file is collected last, so a run that stops at the first
failure has already run every other test; it must also pass on its own in a
fresh process.
"""

import ctypes

import numpy as np
import pytest

from oracle import exl3 as o
from trellis_quantized_linear_rot_gb300 import synth
from helpers import assert_close_f32, dev, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import trellis_quantized_linear_rot_gb300 as tf  # noqa: E402


def _call_noalloc(xr_t, tr_t, svh_t, y_t, bits, rows, i_f, o_f):
    lib = tf.lib()
    return lib.tf_trellis_linear_noalloc(
        ctypes.c_void_p(xr_t.data_ptr()), ctypes.c_void_p(tr_t.data_ptr()),
        ctypes.c_void_p(svh_t.data_ptr()), ctypes.c_void_p(y_t.data_ptr()),
        {torch.float32: tf.TF_F32, torch.float16: tf.TF_F16, torch.bfloat16: tf.TF_BF16}[y_t.dtype],
        rows, i_f, o_f, bits,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("i_f,o_f,bits,rows", [(6144, 25600, 4, 16), (5120, 129280, 4, 1), (384, 256, 6, 17)])
def test_noalloc_matches_regular_entry_point_twice(i_f, o_f, bits, rows):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x = synth.make_x(rows, i_f, 901)
    suh = synth.make_scale(i_f, 902)
    svh = synth.make_scale(o_f, 903)
    tr = synth.make_trellis(i_f, o_f, bits, 904)
    xr_t = tf.tf_rot_in(dev(x), dev(suh))
    tr_t, svh_t = dev(tr), dev(svh)
    want = host(tf.tf_trellis_linear(xr_t, tr_t, svh_t, bits, o_f, out_dtype=torch.float32))
    for _ in range(2):                       # two calls in a row share the array
        y_t = torch.full((rows, o_f), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_noalloc(xr_t, tr_t, svh_t, y_t, bits, rows, i_f, o_f) == tf.TF_OK
        tf.tf_device_error()
        got = host(y_t)
        assert_close_f32(got, want.astype(np.float64), tol=1e-6)
    blocks = [0, o_f // 128 - 1]
    cols = np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])
    ref = o.linear_f64(host(xr_t), o.decode_blocks(tr, i_f, o_f, bits, blocks), svh[cols])
    assert_close_f32(got[:, cols], ref)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_noalloc_mma_kernel_bit_equal_to_tcgen05_kernel(bits):
    """The no-allocation entry point runs every pass on the mma.sync kernel;
    the regular entry point runs the k-tile order on the tcgen05 kernel. Both
    give the same bits for every output, at 1, 8 and 16 rows and at every
    width (2048 -> 8192: several units per CTA and blocks shared between
    CTAs)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    i_f, o_f = 2048, 8192
    tr = synth.make_trellis(i_f, o_f, bits, 910 + bits)
    suh = synth.make_scale(i_f, 920 + bits)
    svh = synth.make_scale(o_f, 930 + bits)
    tr_t, svh_t = dev(tr), dev(svh)
    for rows in (1, 8, 16):
        xr_t = tf.tf_rot_in(dev(synth.make_x(rows, i_f, 940 + rows)), dev(suh))
        want = host(tf.tf_trellis_linear(xr_t, tr_t, svh_t, bits, o_f, out_dtype=torch.float32)).view(np.uint32)
        y_t = torch.full((rows, o_f), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_noalloc(xr_t, tr_t, svh_t, y_t, bits, rows, i_f, o_f) == tf.TF_OK
        tf.tf_device_error()
        got = host(y_t).view(np.uint32)
        assert np.array_equal(got, want), "bits %d, %d rows: the two kernels differ" % (bits, rows)


@pytest.mark.parametrize("rows,out_dtype", [(64, "f32"), (5, "bf16"), (33, "bf16")])
def test_noalloc_many_passes_and_bf16_bit_equal(rows, out_dtype):
    """Several 16-row passes in one call (each pass clears the counters it
    uses and writes its own rows of y) and the bf16 store path: the same bits
    as tf_trellis_linear, on two calls in a row."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    i_f, o_f, bits = 2048, 8192, 4
    dt = {"f32": torch.float32, "bf16": torch.bfloat16}[out_dtype]
    tr_t = dev(synth.make_trellis(i_f, o_f, bits, 960))
    svh_t = dev(synth.make_scale(o_f, 961))
    xr_t = tf.tf_rot_in(dev(synth.make_x(rows, i_f, 962)), dev(synth.make_scale(i_f, 963)))
    want = host(tf.tf_trellis_linear(xr_t, tr_t, svh_t, bits, o_f, out_dtype=dt))
    for _ in range(2):
        y_t = torch.full((rows, o_f), float("nan"), dtype=dt, device="cuda")
        assert _call_noalloc(xr_t, tr_t, svh_t, y_t, bits, rows, i_f, o_f) == tf.TF_OK
        tf.tf_device_error()
        got = host(y_t)
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), "rows %d %s" % (rows, out_dtype)


def test_noalloc_refuses_more_outputs_than_its_array_holds():
    """Shapes tf_trellis_linear refuses get its status; shapes it accepts but
    the fixed array cannot hold get TF_ERR_SCRATCH."""
    lib = tf.lib()
    p = ctypes.c_void_p(0x10000)
    s0 = ctypes.c_void_p(0)
    f = lib.tf_trellis_linear_noalloc
    assert f(p, p, p, p, tf.TF_F32, 1, 512, 128 * 20000, 4, s0) == tf.TF_ERR_SCRATCH
    assert f(p, p, p, p, tf.TF_F32, 1, 512, 2097152 + 128, 4, s0) == tf.TF_ERR_SCRATCH
    assert f(p, p, p, p, tf.TF_F32, 1, 512, (1 << 24) + 128, 4, s0) == tf.TF_ERR_SHAPE
    assert f(p, p, p, p, tf.TF_F32, 1, 512, 100, 4, s0) == tf.TF_ERR_SHAPE
    assert f(p, p, p, p, tf.TF_F32, 1, 512, 128, 7, s0) == tf.TF_ERR_BITS

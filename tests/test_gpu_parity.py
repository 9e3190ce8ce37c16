"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, plus the GPU-vs-GPU invariants the method fixes.

Page: "hip exl3: the input rotation and trellis linear for decode rows"
(TensorFold pull request #3314), sections "What this changes", "Checks on
this head" and "Kernel contract".

Bars: bit-exact for weight decode, rot_in's fp16 outputs, exact-sum cases
(identity rows, gate 4) and row independence; max |y - y_ref| / rms(y_ref
row) <= 1e-4 for fp32 outputs, that plus half an fp16 ulp for fp16 outputs.
"""

import numpy as np
import pytest

from oracle import exl3 as o
from trellis_quantized_linear_rot_gb300 import synth
from helpers import assert_close_bf16, assert_close_f16, assert_close_f32, bits16, dev, dev_bf16, host

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


def inputs(rows, i_f, o_f, bits, c=0):
    x = synth.make_x(rows, i_f, synth.SEED_X + c)
    suh = synth.make_scale(i_f, synth.SEED_SUH + c)
    svh = synth.make_scale(o_f, synth.SEED_SVH + c)
    tr = synth.make_trellis(i_f, o_f, bits, synth.SEED_TRELLIS + c + bits)
    return x, suh, svh, tr


# --------------------------------------------------------------------- rot_in
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("rows,i_f", [(1, 512), (17, 6144), (5, 5120), (3, 128)])
def test_rot_in_bit_exact(dtype, rows, i_f):
    x16 = synth.make_x(rows, i_f, 500 + rows)
    suh = synth.make_scale(i_f, 600 + rows)
    if dtype == "f16":
        x_np, x_t = x16, dev(x16)
    elif dtype == "f32":
        x_np = synth.make_x(rows, i_f, 500 + rows, dtype=np.float32)
        x_t = dev(x_np)
    else:
        x_np = (synth.make_x(rows, i_f, 500 + rows, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
        x_t = dev_bf16(x_np)
    got = host(tf.tf_rot_in(x_t, dev(suh)))
    want = o.rot_in_f32(x_np, suh, dtype)
    assert np.array_equal(bits16(got), bits16(want))


def test_rot_in_non_finite_propagates_through_its_block():
    x = synth.make_x(2, 256, 9)
    x[0, 5] = np.inf
    x[1, 200] = np.nan
    suh = synth.make_scale(256, 10)
    got = host(tf.tf_rot_in(dev(x), dev(suh))).astype(np.float64)
    want = o.rot_in_f32(x, suh).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(np.isinf(got), np.isinf(want))
    assert np.all(np.isfinite(got[0, 128:])) and np.all(np.isfinite(got[1, :128]))


# --------------------------------------------------------------------- decode
@pytest.mark.parametrize("bits", o.BITS_ALLOWED)
def test_decode_bit_exact(bits):
    i_f, o_f = 384, 256
    tr = synth.make_trellis(i_f, o_f, bits, 700 + bits)
    got = host(tf.tf_trellis_decode(dev(tr), i_f, o_f, bits))
    want = o.decode_matrix(tr, i_f, o_f, bits)
    assert np.array_equal(bits16(got), bits16(want))


def test_decode_bit_exact_sampled_head():
    i_f, o_f, bits = 5120, 129280, 4
    tr = synth.make_trellis(i_f, o_f, bits, synth.SEED_TRELLIS + 2 + bits)
    got = host(tf.tf_trellis_decode(dev(tr), i_f, o_f, bits))
    for b in (0, 517, 1009):
        want = o.decode_blocks(tr, i_f, o_f, bits, [b])
        assert np.array_equal(bits16(got[:, 128 * b:128 * b + 128]), bits16(want))


# --------------------------------------------------------------------- linear
def run_linear(xr16, tr, svh, bits, o_f, out_dtype):
    y = tf.tf_trellis_linear(dev(xr16), dev(tr), dev(svh), bits, o_f, out_dtype=out_dtype)
    return host(y)


@pytest.mark.parametrize("bits", o.BITS_ALLOWED)
@pytest.mark.parametrize("rows", [1, 3, 16, 17])
def test_linear_matches_oracle_small(bits, rows):
    i_f, o_f = 384, 256
    x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=10 + rows)
    xr = o.rot_in_f32(x, suh)
    w = o.decode_matrix(tr, i_f, o_f, bits)
    ref = o.linear_f64(xr, w, svh)
    assert_close_f32(run_linear(xr, tr, svh, bits, o_f, torch.float32), ref)
    assert_close_f16(run_linear(xr, tr, svh, bits, o_f, torch.float16), ref)


def test_config_wk_512_to_128_whole_path():
    """wk 512 -> 128, 4 bits, 1 row, fp16 out: rot_in and linear end to end (project: the fused call)."""
    i_f, o_f, bits = 512, 128, 4
    x, suh, svh, tr = inputs(1, i_f, o_f, bits, c=0)
    y = host(tf.project(dev(x), dev(suh), dev(tr), dev(svh), bits, o_f, out_dtype=torch.float16))
    xr, ref = o.project_f64(x, suh, tr, svh, i_f, o_f, bits)
    assert_close_f16(y, ref)


@pytest.mark.parametrize("rows", [1, 4, 16])
def test_config_wkv_sampled(rows):
    """wkv 6144 -> 25,600, 4 bits, fp16 out, rows 1/4/16: sampled output blocks."""
    i_f, o_f, bits = 6144, 25600, 4
    x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=1)
    xr_t = tf.tf_rot_in(dev(x), dev(suh))
    y = host(tf.tf_trellis_linear(xr_t, dev(tr), dev(svh), bits, o_f, out_dtype=torch.float16))
    xr = host(xr_t)
    assert np.array_equal(bits16(xr), bits16(o.rot_in_f32(x, suh)))
    blocks = [0, 77, 199]
    w = o.decode_blocks(tr, i_f, o_f, bits, blocks)
    cols = np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])
    ref = o.linear_f64(xr, w, svh[cols])
    assert_close_f16(y[:, cols], ref)


@pytest.mark.parametrize("rows", [1, 8, 16])
def test_config_head_sampled(rows):
    """LM head 5120 -> 129,280, 4 bits, fp32 logits, rows 1/8/16: sampled blocks."""
    i_f, o_f, bits = 5120, 129280, 4
    x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=2)
    xr_t = tf.tf_rot_in(dev(x), dev(suh))
    y = host(tf.tf_trellis_linear(xr_t, dev(tr), dev(svh), bits, o_f, out_dtype=torch.float32))
    xr = host(xr_t)
    blocks = [0, 1, 500, 1009]
    w = o.decode_blocks(tr, i_f, o_f, bits, blocks)
    cols = np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])
    assert_close_f32(y[:, cols], o.linear_f64(xr, w, svh[cols]))
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("bits", o.BITS_ALLOWED)
def test_config_sweep_identity_rows_bit_exact(bits):
    """wkv 6144 -> 25,600, 8 identity rows (padded with +0): each output row is
    the fp32 epilogue of one decoded weight row, bit for bit."""
    i_f, o_f, rows = 6144, 25600, 8
    tr = synth.make_trellis(i_f, o_f, bits, synth.SEED_TRELLIS + 3 + bits)
    svh = synth.make_scale(o_f, synth.SEED_SVH + 3)
    ks = synth.identity_ks(rows, i_f)
    xr = synth.make_identity_rows(rows, i_f, ks)
    wrows = o.decode_rows(tr, i_f, o_f, bits, ks)
    want32 = o.epilogue_f32(wrows.astype(np.float32), svh)
    y32 = run_linear(xr, tr, svh, bits, o_f, torch.float32)
    assert np.array_equal(y32.view(np.uint32), want32.view(np.uint32))
    y16 = run_linear(xr, tr, svh, bits, o_f, torch.float16)
    assert np.array_equal(bits16(y16), bits16(want32.astype(np.float16)))
    ybf = run_linear(xr, tr, svh, bits, o_f, torch.bfloat16)
    assert np.array_equal(ybf, o.bf16_bits_rne(want32))


@pytest.mark.parametrize("bits,rows", [(4, 1), (4, 16), (2, 5), (8, 17), (6, 3)])
def test_linear_bf16_output(bits, rows):
    """bf16 output: within the bound of the float64 reference, and bit for
    bit the oracle's rounding of the same launch shape's fp32 output."""
    i_f, o_f = 384, 512
    x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=20 + rows)
    xr = o.rot_in_f32(x, suh)
    ref = o.linear_f64(xr, o.decode_matrix(tr, i_f, o_f, bits), svh)
    y32 = run_linear(xr, tr, svh, bits, o_f, torch.float32)
    ybf = run_linear(xr, tr, svh, bits, o_f, torch.bfloat16)
    assert ybf.dtype == np.uint16
    assert np.array_equal(ybf, o.bf16_bits_rne(y32))
    assert_close_bf16(ybf, ref)


def test_config_head_bf16_sampled():
    """LM head 5120 -> 129,280 at 4 bits with bf16 out (the page's bf16-output
    registration of the linear), 1 row: sampled blocks."""
    i_f, o_f, bits = 5120, 129280, 4
    x, suh, svh, tr = inputs(1, i_f, o_f, bits, c=2)
    xr_t = tf.tf_rot_in(dev(x), dev(suh))
    y = host(tf.tf_trellis_linear(xr_t, dev(tr), dev(svh), bits, o_f, out_dtype=torch.bfloat16))
    blocks = [0, 640, 1009]
    w = o.decode_blocks(tr, i_f, o_f, bits, blocks)
    cols = np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])
    assert_close_bf16(y[:, cols], o.linear_f64(host(xr_t), w, svh[cols]))


@pytest.mark.parametrize("bits", o.BITS_ALLOWED)
def test_config_sweep_random_rows(bits):
    """wkv 6144 -> 25,600, 8 random rows, every width, fp16 out: sampled blocks."""
    i_f, o_f, rows = 6144, 25600, 8
    x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=3)
    xr = o.rot_in_f32(x, suh)
    y = run_linear(xr, tr, svh, bits, o_f, torch.float16)
    blocks = [3, 150]
    cols = np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])
    ref = o.linear_f64(xr, o.decode_blocks(tr, i_f, o_f, bits, blocks), svh[cols])
    assert_close_f16(y[:, cols], ref)


def test_gate4_exact_sums():
    """All-ones trellis, xr = 4096, in = 6144: exact integer sums; 127 exact
    zeros per block after the rotation; fp16 output overflows to -inf*sign."""
    i_f, o_f, bits = 6144, 256, 4
    tr = synth.make_trellis_all_ones(i_f, o_f, bits)
    svh = synth.make_scale(o_f, 91)
    xr = np.full((3, i_f), np.float16(4096.0))
    acc = np.full((3, o_f), np.float32(-16392192.0))
    want = o.epilogue_f32(acc, svh)
    y32 = run_linear(xr, tr, svh, bits, o_f, torch.float32)
    assert np.array_equal(y32.view(np.uint32), want.view(np.uint32))
    assert np.sum(y32[0, :128] == 0.0) == 127
    y16 = run_linear(xr, tr, svh, bits, o_f, torch.float16).astype(np.float64)
    for b in range(o_f // 128):
        assert np.isinf(y16[0, 128 * b]) and np.sign(y16[0, 128 * b]) == -np.sign(float(svh[128 * b]))
    # bf16 has fp32's range: no overflow, one rounding of the exact fp32 values.
    ybf = run_linear(xr, tr, svh, bits, o_f, torch.bfloat16)
    assert np.array_equal(ybf, o.bf16_bits_rne(want))


def test_non_finite_classes_match_float64():
    i_f, o_f, bits = 256, 256, 4
    x, suh, svh, tr = inputs(2, i_f, o_f, bits, c=4)
    xr = o.rot_in_f32(x, suh)
    xr[0, 3] = np.float16(np.inf)
    xr[1, 200] = np.float16(np.nan)
    y = run_linear(xr, tr, svh, bits, o_f, torch.float32).astype(np.float64)
    ref = o.linear_f64(xr, o.decode_matrix(tr, i_f, o_f, bits), svh)
    assert np.array_equal(np.isnan(y), np.isnan(ref))
    assert np.array_equal(np.isposinf(y), np.isposinf(ref))
    assert np.array_equal(np.isneginf(y), np.isneginf(ref))


# -------------------------------------------------------------- maximum sizes
def test_max_in_features_one_block_across_every_cta():
    """in = 2^20 (the largest accepted), out = 128, 3 rows, 4 bits: the one
    output block is cut between every CTA of the launch, whose partial sums
    the last arriver adds in CTA order. Each row of xr is zero except at 96
    random inputs spread over the whole range (and the first and last), so
    every CTA's part carries terms while the float64 reference needs only
    those weight rows; the kernel still streams and decodes all weights."""
    i_f, o_f, bits, rows = 1 << 20, 128, 4, 3
    g = np.random.Generator(np.random.PCG64(4321))
    tr = synth.make_trellis(i_f, o_f, bits, synth.SEED_TRELLIS + 30 + bits)
    svh = synth.make_scale(o_f, synth.SEED_SVH + 30)
    xr = np.zeros((rows, i_f), np.float16)
    ks = np.unique(np.concatenate([[0, i_f - 1], g.integers(0, i_f, size=96)]))
    for r in range(rows):
        xr[r, ks] = g.standard_normal(ks.size).astype(np.float16)
    y = run_linear(xr, tr, svh, bits, o_f, torch.float32)
    # The zero inputs add nothing: the reference is the oracle's linear over
    # the chosen inputs and their decoded weight rows.
    ref = o.linear_f64(xr[:, ks], o.decode_rows(tr, i_f, o_f, bits, ks), svh)
    assert_close_f32(y, ref)


def test_max_out_features_sampled():
    """out = 2^24 (the largest accepted), in = 128, 1 row, 2 bits, fp16 out:
    131,072 output blocks; sampled blocks at both ends and the middle."""
    i_f, o_f, bits = 128, 1 << 24, 2
    x, suh, svh, tr = inputs(1, i_f, o_f, bits, c=31)
    xr = o.rot_in_f32(x, suh)
    y = run_linear(xr, tr, svh, bits, o_f, torch.float16)
    blocks = [0, 65536, (o_f // 128) - 1]
    cols = np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])
    ref = o.linear_f64(xr, o.decode_blocks(tr, i_f, o_f, bits, blocks), svh[cols])
    assert_close_f16(y[:, cols], ref)


# ------------------------------------------------------------ strips layout
@pytest.mark.parametrize("bits", o.BITS_ALLOWED)
def test_to_strips_matches_oracle_order(bits):
    i_f, o_f = 384, 256
    tr = synth.make_trellis(i_f, o_f, bits, 800 + bits)
    got = host(tf.tf_trellis_to_strips(dev(tr), i_f, o_f, bits)).view(np.uint32)
    assert np.array_equal(got, o.tiles_to_strips(tr, i_f, o_f, bits))


@pytest.mark.parametrize("bits,rows", [(4, 1), (4, 16), (6, 9), (8, 3), (3, 16), (2, 5), (5, 12),
                                       (4, 32), (6, 24), (2, 17), (8, 29), (5, 40)])
def test_linear_strips_equals_tiles_bit_for_bit(bits, rows):
    """The strips order streams the same tiles: outputs are identical bits,
    and match the oracle (sampled) on the wkv shape."""
    i_f, o_f = 6144, 25600
    x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=7)
    xr_t, tr_t, svh_t = dev(o.rot_in_f32(x, suh)), dev(tr), dev(svh)
    strips_t = tf.tf_trellis_to_strips(tr_t, i_f, o_f, bits)
    a = host(tf.tf_trellis_linear(xr_t, tr_t, svh_t, bits, o_f, out_dtype=torch.float32))
    b = host(tf.tf_trellis_linear_strips(xr_t, strips_t, svh_t, bits, o_f, out_dtype=torch.float32))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    blocks = [5, 123]
    cols = np.concatenate([np.arange(128 * bl, 128 * bl + 128) for bl in blocks])
    ref = o.linear_f64(host(xr_t), o.decode_blocks(tr, i_f, o_f, bits, blocks), svh[cols])
    assert_close_f32(b[:, cols], ref)


# ------------------------------------------------------- GPU-vs-GPU invariants
@pytest.mark.parametrize("layout", ["tiles", "strips"])
def test_row_independence_windows_and_passes(layout):
    """LM head 5120 -> 129,280 at 6 bits, 64 rows in one pass (the tcgen05
    kernel): every row's outputs equal its single-row run (the mma.sync
    kernel) bit for bit, also inside random windows of 2 to 24 rows, which
    run on either kernel ("Checks on this head", the window test), in both
    weight orders."""
    i_f, o_f, bits, rows = 5120, 129280, 6, 64
    x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=5)
    tr_t, svh_t = dev(tr), dev(svh)
    lin = tf.tf_trellis_linear
    if layout == "strips":
        tr_t = tf.tf_trellis_to_strips(tr_t, i_f, o_f, bits)
        lin = tf.tf_trellis_linear_strips
    xr_t = tf.tf_rot_in(dev(x), dev(suh))
    full = host(lin(xr_t, tr_t, svh_t, bits, o_f, out_dtype=torch.float32)).view(np.uint32)
    singles = {}
    for r in range(rows):
        singles[r] = host(lin(xr_t[r:r + 1], tr_t, svh_t, bits, o_f,
                              out_dtype=torch.float32)).view(np.uint32)[0]
        assert np.array_equal(full[r], singles[r]), "row %d differs in the 64-row launch" % r
    for first, n in synth.random_windows(rows, 50, seed=55):
        win = host(lin(xr_t[first:first + n], tr_t, svh_t, bits, o_f,
                       out_dtype=torch.float32)).view(np.uint32)
        for j in range(n):
            assert np.array_equal(win[j], singles[first + j]), "window (%d, %d) row %d" % (first, n, j)
    blocks = [2, 700]
    cols = np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])
    ref = o.linear_f64(host(xr_t), o.decode_blocks(tr, i_f, o_f, bits, blocks), svh[cols])
    assert_close_f32(full.view(np.float32)[:, cols], ref)


def test_five_runs_byte_identical():
    i_f, o_f, bits = 6144, 25600, 4
    x, suh, svh, tr = inputs(16, i_f, o_f, bits, c=6)
    xr_t, tr_t, svh_t = dev(o.rot_in_f32(x, suh)), dev(tr), dev(svh)
    outs = [host(tf.tf_trellis_linear(xr_t, tr_t, svh_t, bits, o_f, out_dtype=torch.float32)).tobytes()
            for _ in range(5)]
    assert all(b == outs[0] for b in outs)


def test_empty_batch_is_a_no_op():
    y = torch.full((0, 128), 7.0, device="cuda")
    tf.tf_trellis_linear(torch.empty((0, 512), dtype=torch.float16, device="cuda"),
                         dev(synth.make_trellis(512, 128, 4, 1)), dev(synth.make_scale(128, 2)), 4, 128, y=y)
    tf.tf_device_error()


def test_host_pointer_is_refused():
    xr = torch.zeros((1, 512), dtype=torch.float16)   # host memory
    with pytest.raises(tf.TFError) as e:
        tf.tf_trellis_linear(xr, dev(synth.make_trellis(512, 128, 4, 1)), dev(synth.make_scale(128, 2)),
                             4, 128, y=torch.empty((1, 128), device="cuda"))
    assert e.value.status == tf.TF_ERR_POINTER


# ------------------------------------------------------------- prompt passes
@pytest.mark.parametrize("bits,rows,layout", [(4, 17, "strips"), (6, 32, "tiles"), (4, 33, "tiles"),
                                              (4, 128, "strips"), (6, 100, "tiles"), (2, 129, "strips"),
                                              (8, 64, "strips"), (3, 200, "tiles"), (5, 96, "strips")])
def test_prompt_pass_rows_bit_equal_to_decode_rows(bits, rows, layout):
    """Passes of 17 to 200 rows (up to 128 per pass, on the tcgen05 kernel)
    give every row the same bits as its run alone and as its 16-row pass
    (on whichever kernel the dispatch picks for those), and match the
    oracle; wkv shape 6144 -> 25,600."""
    i_f, o_f = 6144, 25600
    x, suh, svh, tr = inputs(rows, i_f, o_f, bits, c=60 + bits)
    tr_t, svh_t = dev(tr), dev(svh)
    lin = tf.tf_trellis_linear
    if layout == "strips":
        tr_t = tf.tf_trellis_to_strips(tr_t, i_f, o_f, bits)
        lin = tf.tf_trellis_linear_strips
    xr_t = tf.tf_rot_in(dev(x), dev(suh))
    full = host(lin(xr_t, tr_t, svh_t, bits, o_f, out_dtype=torch.float32)).view(np.uint32)
    for r0 in range(0, rows, 16):
        part = host(lin(xr_t[r0:r0 + 16], tr_t, svh_t, bits, o_f, out_dtype=torch.float32)).view(np.uint32)
        assert np.array_equal(full[r0:r0 + 16], part), "rows %d.. differ from their 16-row pass" % r0
    for r in (0, rows // 2, rows - 1):
        one = host(lin(xr_t[r:r + 1], tr_t, svh_t, bits, o_f, out_dtype=torch.float32)).view(np.uint32)
        assert np.array_equal(full[r], one[0])
    blocks = [0, 123, 199]
    cols = np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])
    ref = o.linear_f64(host(xr_t), o.decode_blocks(tr, i_f, o_f, bits, blocks), svh[cols])
    assert_close_f32(full.view(np.float32)[:, cols], ref)


def test_prompt_pass_low_precision_outputs_and_identity():
    """A 48-row pass with fp16 and bf16 outputs equals the oracle's rounding of
    its own fp32 output; identity rows are the decoded weight rows' epilogue,
    bit for bit."""
    i_f, o_f, bits, rows = 6144, 25600, 4, 48
    tr = synth.make_trellis(i_f, o_f, bits, synth.SEED_TRELLIS + 70)
    svh = synth.make_scale(o_f, synth.SEED_SVH + 70)
    ks = synth.identity_ks(rows, i_f)
    xr = synth.make_identity_rows(rows, i_f, ks)
    want32 = o.epilogue_f32(o.decode_rows(tr, i_f, o_f, bits, ks).astype(np.float32), svh)
    y32 = run_linear(xr, tr, svh, bits, o_f, torch.float32)
    assert np.array_equal(y32.view(np.uint32), want32.view(np.uint32))
    y16 = run_linear(xr, tr, svh, bits, o_f, torch.float16)
    assert np.array_equal(bits16(y16), bits16(want32.astype(np.float16)))
    ybf = run_linear(xr, tr, svh, bits, o_f, torch.bfloat16)
    assert np.array_equal(ybf, o.bf16_bits_rne(want32))


# ------------------------------------------------------------ caller workspace
def test_linear_ws_concurrent_streams_match_serial_calls():
    """Two calls on two streams at once, each with its own workspace, give the
    same bits as tf_trellis_linear one after the other (tiles and strips); a
    workspace one byte short is refused."""
    i_f, o_f, bits = 6144, 25600, 4
    xa, suh, svh, tr = inputs(3, i_f, o_f, bits, c=50)
    xb = synth.make_x(20, i_f, 51)
    tr_t, svh_t = dev(tr), dev(svh)
    st_t = tf.tf_trellis_to_strips(tr_t, i_f, o_f, bits)
    xra = tf.tf_rot_in(dev(xa), dev(suh))
    xrb = tf.tf_rot_in(dev(xb), dev(suh))
    ref_a = host(tf.tf_trellis_linear(xra, tr_t, svh_t, bits, o_f, out_dtype=torch.float32))
    ref_b = host(tf.tf_trellis_linear(xrb, tr_t, svh_t, bits, o_f, out_dtype=torch.float32))
    need = tf.tf_trellis_workspace_bytes(i_f, o_f, bits)
    assert need > 0
    wa = torch.empty(need, dtype=torch.uint8, device="cuda")
    wb = torch.empty(need, dtype=torch.uint8, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for layout, w in (("tiles", tr_t), ("strips", st_t)):
        ya = torch.empty((3, o_f), dtype=torch.float32, device="cuda")
        yb = torch.empty((20, o_f), dtype=torch.float32, device="cuda")
        for _ in range(3):
            tf.tf_trellis_linear_ws(xra, w, svh_t, bits, o_f, wa, layout=layout, y=ya, stream=sa)
            tf.tf_trellis_linear_ws(xrb, w, svh_t, bits, o_f, wb, layout=layout, y=yb, stream=sb)
        torch.cuda.synchronize()
        tf.tf_device_error()
        assert np.array_equal(host(ya).view(np.uint32), ref_a.view(np.uint32))
        assert np.array_equal(host(yb).view(np.uint32), ref_b.view(np.uint32))
    with pytest.raises(tf.TFError) as err:
        tf.tf_trellis_linear_ws(xra, tr_t, svh_t, bits, o_f, wa[:need - 1])
    assert err.value.status == tf.TF_ERR_SCRATCH


# ------------------------------------------------------------- failure path
def test_stranded_wait_reports_timeout_and_context_survives():
    """A kernel whose barrier wait nothing completes gives up after the
    bounded-wait limit, the host reads TF_ERR_TIMEOUT, and the context goes
    on working (a linear right after it matches the oracle)."""
    tf.tf_device_error()
    tf.tf_selftest_stranded_wait()
    with pytest.raises(tf.TFError) as err:
        tf.tf_device_error()
    assert err.value.status == tf.TF_ERR_TIMEOUT
    tf.tf_device_error()  # the record was cleared
    i_f, o_f, bits = 384, 256, 4
    x, suh, svh, tr = inputs(2, i_f, o_f, bits, c=40)
    xr = o.rot_in_f32(x, suh)
    y = run_linear(xr, tr, svh, bits, o_f, torch.float32)
    tf.tf_device_error()
    assert_close_f32(y, o.linear_f64(xr, o.decode_matrix(tr, i_f, o_f, bits), svh))

"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point the public header declares, and refuses bad arguments with
the documented status before it makes any CUDA call."""

import ctypes
import os
import re

import pytest

import trellis_quantized_linear_rot_gb300 as tf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(tf_[a-z0-9_]+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(tf.library_path()):
        from trellis_quantized_linear_rot_gb300 import build
        build.build()
    return tf.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"tf_rot_in", "tf_trellis_linear", "tf_trellis_bytes", "tf_status_string"} <= names
    raw = ctypes.CDLL(tf.library_path())
    for n in sorted(names):
        assert hasattr(raw, n), n
    assert names == set(tf.SIGNATURES), "binding and header disagree"


def test_abi_version_and_status_strings(lib):
    assert lib.tf_abi_version() == 1
    for s in range(10):
        assert lib.tf_status_string(s).decode() not in ("", "unknown status")
    assert lib.tf_status_string(99).decode() == "unknown status"


@pytest.mark.parametrize("i,o,b,want", [
    (5120, 129280, 4, 5120 * 129280 // 2), (6144, 25600, 3, 6144 * 25600 * 3 // 8),
    (512, 128, 8, 512 * 128), (512, 128, 7, 0), (100, 128, 4, 0), (128, 0, 4, 0), (-128, 128, 4, 0)])
def test_trellis_bytes(lib, i, o, b, want):
    assert lib.tf_trellis_bytes(i, o, b) == want


P = ctypes.c_void_p(0x10000)      # aligned, non-null, never dereferenced by a refused call
MIS = ctypes.c_void_p(0x10008)    # 8-byte aligned only
NUL = ctypes.c_void_p(0)
S = ctypes.c_void_p(0)


def lin(lib, xr=P, tr=P, svh=P, y=P, dt=tf.TF_F32, rows=1, i=512, o=128, bits=4):
    return lib.tf_trellis_linear(xr, tr, svh, y, dt, rows, i, o, bits, S)


def test_linear_refusals(lib):
    assert lin(lib, rows=-1) == tf.TF_ERR_SHAPE
    assert lin(lib, i=500) == tf.TF_ERR_SHAPE
    assert lin(lib, o=0) == tf.TF_ERR_SHAPE
    assert lin(lib, i=-128) == tf.TF_ERR_SHAPE
    assert lin(lib, bits=7) == tf.TF_ERR_BITS
    assert lin(lib, bits=1) == tf.TF_ERR_BITS
    # bf16 output is accepted (the refusal then comes from the NULL buffer);
    # any other code is not.
    assert lin(lib, dt=tf.TF_BF16, xr=NUL) == tf.TF_ERR_NULL
    assert lin(lib, dt=3) == tf.TF_ERR_DTYPE
    assert lin(lib, dt=9) == tf.TF_ERR_DTYPE
    assert lin(lib, xr=NUL) == tf.TF_ERR_NULL
    assert lin(lib, tr=NUL) == tf.TF_ERR_NULL
    assert lin(lib, y=NUL) == tf.TF_ERR_NULL
    assert lin(lib, tr=MIS) == tf.TF_ERR_ALIGN
    assert lin(lib, svh=MIS) == tf.TF_ERR_ALIGN
    # An empty batch is valid and touches nothing, even with NULL buffers.
    assert lin(lib, rows=0, xr=NUL, y=NUL) == tf.TF_OK


def test_linear_ws_refusals(lib):
    f = lib.tf_trellis_linear_ws
    def ws(layout=0, work=P, rows=1, i=512, bits=4, dt=tf.TF_F32):
        return f(P, P, P, P, dt, rows, i, 128, bits, layout, work, 1 << 20, S)
    assert ws(layout=2) == tf.TF_ERR_SHAPE
    assert ws(i=500) == tf.TF_ERR_SHAPE
    assert ws(bits=7) == tf.TF_ERR_BITS
    assert ws(dt=5) == tf.TF_ERR_DTYPE
    assert ws(work=NUL) == tf.TF_ERR_NULL
    assert ws(work=ctypes.c_void_p(0x10010)) == tf.TF_ERR_ALIGN   # 16-byte aligned only
    assert ws(rows=0, work=NUL) == tf.TF_OK
    assert lib.tf_trellis_workspace_bytes(500, 128, 4) == 0


def test_rot_in_refusals(lib):
    f = lib.tf_rot_in
    assert f(P, tf.TF_F16, P, P, -1, 512, S) == tf.TF_ERR_SHAPE
    assert f(P, tf.TF_F16, P, P, 1, 130, S) == tf.TF_ERR_SHAPE
    assert f(P, 7, P, P, 1, 512, S) == tf.TF_ERR_DTYPE
    assert f(NUL, tf.TF_F16, P, P, 1, 512, S) == tf.TF_ERR_NULL
    assert f(P, tf.TF_F16, P, MIS, 1, 512, S) == tf.TF_ERR_ALIGN
    assert f(NUL, tf.TF_F16, NUL, NUL, 0, 512, S) == tf.TF_OK


@pytest.mark.parametrize("name", ["tf_rot_in_linear", "tf_rot_in_linear_strips"])
def test_rot_in_linear_refusals(lib, name):
    f = getattr(lib, name)
    def call(x=P, xdt=tf.TF_F16, suh=P, xr=P, tr=P, svh=P, y=P, dt=tf.TF_F32, rows=1, i=512, o=128, bits=4):
        return f(x, xdt, suh, xr, tr, svh, y, dt, rows, i, o, bits, S)
    assert call(rows=-1) == tf.TF_ERR_SHAPE
    assert call(i=500) == tf.TF_ERR_SHAPE
    assert call(o=0) == tf.TF_ERR_SHAPE
    assert call(bits=7) == tf.TF_ERR_BITS
    assert call(xdt=7) == tf.TF_ERR_DTYPE
    assert call(dt=3) == tf.TF_ERR_DTYPE
    for k in ("x", "suh", "xr", "tr", "svh", "y"):
        assert call(**{k: NUL}) == tf.TF_ERR_NULL, k
        assert call(**{k: MIS}) == tf.TF_ERR_ALIGN, k
    assert call(rows=0, x=NUL, xr=NUL, y=NUL) == tf.TF_OK


def test_decode_refusals(lib):
    f = lib.tf_trellis_decode
    assert f(P, P, 512, 100, 4, S) == tf.TF_ERR_SHAPE
    assert f(P, P, 512, 128, 9, S) == tf.TF_ERR_BITS
    assert f(NUL, P, 512, 128, 4, S) == tf.TF_ERR_NULL
    assert f(P, MIS, 512, 128, 4, S) == tf.TF_ERR_ALIGN


def test_without_gpu_a_valid_call_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lin(lib) in (tf.TF_ERR_CUDA, tf.TF_ERR_POINTER)
    assert "" != lib.tf_last_error().decode() or True


PAGE_SECTIONS = ("What this changes", "Checks on this head", "Kernel contract", "Known limits")


def comment_before_each_declaration():
    """(function name, the comment block right before its declaration) for
    every function the public headers declare."""
    out = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        pattern = r"/\*((?:(?!\*/).)*)\*/\s*((?:const\s+)?[a-z_0-9]+\s*\*?\s*)(tf_[a-z0-9_]+)\s*\("
        for m in re.finditer(pattern, text, re.S):
            out.append((m.group(3), m.group(1)))
    return out


def test_every_entry_point_cites_a_passage_or_says_it_has_none():
    """Each declaration's comment names the page section it follows (quoted)
    or says that the pages have no counterpart."""
    found = comment_before_each_declaration()
    assert {n for n, _ in found} == declared_functions()
    for name, comment in found:
        flat = " ".join(comment.replace("*", " ").split())
        cites = any('"%s"' % sec in flat or "%s," % sec in flat for sec in PAGE_SECTIONS)
        assert cites or "no counterpart" in flat, name

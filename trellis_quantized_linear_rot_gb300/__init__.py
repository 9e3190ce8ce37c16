"""GB300 (sm_103a) trellis-quantized projection for decode rows.

A thin Python binding over the C ABI of libtf_exl3.so (include/tf_exl3.h),
with the same names. It only marshals arguments: every step of the
computation runs in the library's CUDA kernels. PyTorch provides device
memory and streams. There is no CPU fallback: a missing library raises.

Method: "hip exl3: the input rotation and trellis linear for decode rows"
(TensorFold pull request #3314), section "What this changes".
"""

import ctypes
import os

from . import build as _build

TF_OK, TF_ERR_NULL, TF_ERR_SHAPE, TF_ERR_BITS, TF_ERR_DTYPE = 0, 1, 2, 3, 4
TF_ERR_ALIGN, TF_ERR_CUDA, TF_ERR_TIMEOUT, TF_ERR_POINTER, TF_ERR_SCRATCH = 5, 6, 7, 8, 9
TF_F16, TF_F32, TF_BF16 = 0, 1, 2

# Every entry point include/tf_exl3.h declares, with its ctypes signature.
_VP, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "tf_abi_version": (_I, []),
    "tf_rot_in": (_I, [_VP, _I, _VP, _VP, _I, _I, _VP]),
    "tf_trellis_linear": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP]),
    "tf_rot_in_linear": (_I, [_VP, _I, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP]),
    "tf_rot_in_linear_strips": (_I, [_VP, _I, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP]),
    "tf_trellis_linear_noalloc": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP]),
    "tf_trellis_linear_strips": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP]),
    "tf_trellis_to_strips": (_I, [_VP, _VP, _I, _I, _I, _VP]),
    "tf_trellis_workspace_bytes": (_SZ, [_I, _I, _I]),
    "tf_trellis_linear_ws": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP, _SZ, _VP]),
    "tf_trellis_decode": (_I, [_VP, _VP, _I, _I, _I, _VP]),
    "tf_trellis_bytes": (_SZ, [_I, _I, _I]),
    "tf_status_string": (ctypes.c_char_p, [_I]),
    "tf_last_error": (ctypes.c_char_p, []),
    "tf_device_error": (_I, [_VP]),
    "tf_selftest_stranded_wait": (_I, [_VP]),
}

_lib = None


class TFError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s: %s (status %d)%s" % (what, lib().tf_status_string(status).decode(), status,
                                                    _cuda_detail(status)))


def _cuda_detail(status):
    if status == TF_ERR_CUDA:
        return ": " + lib().tf_last_error().decode()
    return ""


def library_path():
    return _build.LIB_PATH


def lib():
    """The loaded C library. Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError("libtf_exl3.so is not built (run __graft_entry__.build()); "
                               "this package has no CPU fallback")
        handle = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status, what):
    if status != TF_OK:
        raise TFError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt):
    import torch
    codes = {torch.float16: TF_F16, torch.float32: TF_F32, torch.bfloat16: TF_BF16}
    if dt not in codes:
        raise TypeError("unsupported dtype %s" % dt)
    return codes[dt]


def _contig(t, name):
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def tf_trellis_bytes(in_features, out_features, bits):
    return lib().tf_trellis_bytes(in_features, out_features, bits)


def tf_status_string(status):
    return lib().tf_status_string(status).decode()


def tf_abi_version():
    return lib().tf_abi_version()


def tf_rot_in(x, suh, xr=None, stream=None):
    """xr = fp16 rows of x * suh rotated by 128 (see tf_rot_in in tf_exl3.h).

    x: [rows, in] fp16/bf16/fp32 CUDA tensor; suh: [in] fp16. Returns xr.
    """
    import torch
    rows, in_f = x.shape
    _contig(x, "x")
    _contig(suh, "suh")
    if xr is None:
        xr = torch.empty((rows, in_f), dtype=torch.float16, device=x.device)
    _contig(xr, "xr")
    st = lib().tf_rot_in(_ptr(x), _dtype_code(x.dtype), _ptr(suh), _ptr(xr), rows, in_f, _stream(stream))
    _check(st, "tf_rot_in")
    return xr


def tf_trellis_linear(xr, trellis, svh, bits, out_features, out_dtype=None, y=None, stream=None):
    """y = trellis linear of the rotated rows xr (see tf_trellis_linear).

    xr: [rows, in] fp16; trellis: packed uint32 words (torch.int32 storage);
    svh: [out] fp16; out_dtype torch.float16, torch.float32 or torch.bfloat16.
    Returns y.
    """
    import torch
    rows, in_f = xr.shape
    for t, n in ((xr, "xr"), (trellis, "trellis"), (svh, "svh")):
        _contig(t, n)
    if y is None:
        y = torch.empty((rows, out_features), dtype=out_dtype or torch.float32, device=xr.device)
    _contig(y, "y")
    st = lib().tf_trellis_linear(_ptr(xr), _ptr(trellis), _ptr(svh), _ptr(y), _dtype_code(y.dtype), rows,
                                 in_f, out_features, bits, _stream(stream))
    _check(st, "tf_trellis_linear")
    return y


def tf_rot_in_linear(x, suh, trellis, svh, bits, out_features, out_dtype=None, xr=None, y=None, stream=None,
                     strips=False):
    """tf_rot_in then tf_trellis_linear in one launch per pass (see tf_rot_in_linear).

    x: [rows, in] fp16/bf16/fp32; suh: [in] fp16; trellis in the k-tile-major
    order (strips=True: the strips order, tf_rot_in_linear_strips); svh: [out]
    fp16. xr (written, [rows, in] fp16) and y are allocated when not given.
    Returns (xr, y).
    """
    import torch
    rows, in_f = x.shape
    for t, n in ((x, "x"), (suh, "suh"), (trellis, "trellis"), (svh, "svh")):
        _contig(t, n)
    if xr is None:
        xr = torch.empty((rows, in_f), dtype=torch.float16, device=x.device)
    if y is None:
        y = torch.empty((rows, out_features), dtype=out_dtype or torch.float32, device=x.device)
    _contig(xr, "xr")
    _contig(y, "y")
    f = lib().tf_rot_in_linear_strips if strips else lib().tf_rot_in_linear
    st = f(_ptr(x), _dtype_code(x.dtype), _ptr(suh), _ptr(xr), _ptr(trellis), _ptr(svh), _ptr(y),
           _dtype_code(y.dtype), rows, in_f, out_features, bits, _stream(stream))
    _check(st, "tf_rot_in_linear_strips" if strips else "tf_rot_in_linear")
    return xr, y


def tf_trellis_linear_strips(xr, strips, svh, bits, out_features, out_dtype=None, y=None, stream=None):
    """tf_trellis_linear on weights stored in the strips order (tf_trellis_to_strips)."""
    import torch
    rows, in_f = xr.shape
    for t, n in ((xr, "xr"), (strips, "strips"), (svh, "svh")):
        _contig(t, n)
    if y is None:
        y = torch.empty((rows, out_features), dtype=out_dtype or torch.float32, device=xr.device)
    _contig(y, "y")
    st = lib().tf_trellis_linear_strips(_ptr(xr), _ptr(strips), _ptr(svh), _ptr(y), _dtype_code(y.dtype),
                                        rows, in_f, out_features, bits, _stream(stream))
    _check(st, "tf_trellis_linear_strips")
    return y


def tf_trellis_workspace_bytes(in_features, out_features, bits):
    return lib().tf_trellis_workspace_bytes(in_features, out_features, bits)


def tf_trellis_linear_ws(xr, trellis, svh, bits, out_features, workspace, layout="tiles", out_dtype=None,
                         y=None, stream=None):
    """The trellis linear with its scratch in `workspace` (a CUDA tensor of at
    least tf_trellis_workspace_bytes bytes); layout "tiles" or "strips"."""
    import torch
    rows, in_f = xr.shape
    for t, n in ((xr, "xr"), (trellis, "trellis"), (svh, "svh"), (workspace, "workspace")):
        _contig(t, n)
    if y is None:
        y = torch.empty((rows, out_features), dtype=out_dtype or torch.float32, device=xr.device)
    _contig(y, "y")
    nbytes = workspace.numel() * workspace.element_size()
    st = lib().tf_trellis_linear_ws(_ptr(xr), _ptr(trellis), _ptr(svh), _ptr(y), _dtype_code(y.dtype), rows,
                                    in_f, out_features, bits, {"tiles": 0, "strips": 1}[layout],
                                    _ptr(workspace), nbytes, _stream(stream))
    _check(st, "tf_trellis_linear_ws")
    return y


def tf_trellis_to_strips(tiles, in_features, out_features, bits, strips=None, stream=None):
    """Repacks k-tile-major packed tiles into the strips order."""
    import torch
    _contig(tiles, "tiles")
    if strips is None:
        strips = torch.empty_like(tiles)
    st = lib().tf_trellis_to_strips(_ptr(tiles), _ptr(strips), in_features, out_features, bits,
                                    _stream(stream))
    _check(st, "tf_trellis_to_strips")
    return strips


def tf_trellis_decode(trellis, in_features, out_features, bits, w=None, stream=None):
    """Dense fp16 W [in, out] decoded from the packed trellis."""
    import torch
    _contig(trellis, "trellis")
    if w is None:
        w = torch.empty((in_features, out_features), dtype=torch.float16, device=trellis.device)
    st = lib().tf_trellis_decode(_ptr(trellis), _ptr(w), in_features, out_features, bits, _stream(stream))
    _check(st, "tf_trellis_decode")
    return w


def tf_selftest_stranded_wait(stream=None):
    """Launches the failure-path self-test (see tf_selftest_stranded_wait)."""
    _check(lib().tf_selftest_stranded_wait(_stream(stream)), "tf_selftest_stranded_wait")


def tf_device_error(stream=None):
    """Synchronises the stream; raises TFError if a kernel gave up a bounded wait."""
    _check(lib().tf_device_error(_stream(stream)), "tf_device_error")


def project(x, suh, trellis, svh, bits, out_features, out_dtype=None, stream=None):
    """The whole decode-row projection (weights in the k-tile-major order), as
    one fused call: the bits of tf_rot_in then tf_trellis_linear, one launch
    per pass. Returns y."""
    return tf_rot_in_linear(x, suh, trellis, svh, bits, out_features, out_dtype=out_dtype, stream=stream)[1]

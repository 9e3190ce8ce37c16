"""Shared test helpers: device transfer of numpy arrays and the tolerance
checks the parity tests apply."""

import numpy as np


def dev(a):
    """numpy array -> CUDA tensor with the same bits (uint32 kept as int32,
    a uint16 array tagged 'bf16' becomes bfloat16)."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def dev_bf16(bits16):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits16).view(np.int16)).cuda().view(torch.bfloat16)


def host(t):
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bits16(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


REL_TOL = 1e-4   # max |y - y_ref| / rms(y_ref row)


def rel_err_rows(y, y_ref):
    """Per row: max |y - y_ref| / rms(y_ref row), on finite references."""
    y = np.asarray(y, dtype=np.float64)
    rms = np.sqrt(np.mean(np.square(y_ref), axis=1))
    return np.max(np.abs(y - y_ref), axis=1) / rms


def assert_close_f32(y, y_ref, tol=REL_TOL):
    err = rel_err_rows(y, y_ref)
    assert np.all(err <= tol), "worst relative error %.3e > %.1e (row %d)" % (err.max(), tol, err.argmax())
    return float(err.max())


def assert_close_f16(y16, y_ref, tol=REL_TOL):
    """fp16 outputs: the fp32 value may be off by tol * rms(row), then one
    rounding to fp16 adds at most half an fp16 ulp of the rounded value."""
    y = np.asarray(y16, dtype=np.float16)
    rms = np.sqrt(np.mean(np.square(y_ref), axis=1))[:, None]
    slack = tol * rms
    with np.errstate(over="ignore"):
        hi = (np.abs(y_ref) + slack).astype(np.float16)
    half_ulp = 0.5 * np.spacing(hi).astype(np.float64)
    yf = y.astype(np.float64)
    ok_inf = np.isinf(yf) & (np.abs(y_ref) >= 65504.0)
    err = np.abs(yf - y_ref)
    good = (err <= slack + half_ulp) | ok_inf
    assert np.all(good), "fp16 output outside bound at %s" % (np.argwhere(~good)[:5].tolist(),)
    return float(np.max(np.where(np.isfinite(err), err / np.maximum(rms, 1e-300), 0.0)))


def bf16_to_f64(bits):
    """bf16 bit patterns (uint16) -> float64 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close_bf16(ybits, y_ref, tol=REL_TOL):
    """bf16 outputs (uint16 bit patterns): the fp32 value may be off by
    tol * rms(row); one rounding to bf16 (8 significant bits) then adds at most
    half a bf16 place of the value, i.e. 2^(e - 9) for a value in
    [2^(e-1), 2^e)."""
    y = bf16_to_f64(ybits)
    rms = np.sqrt(np.mean(np.square(y_ref), axis=1))[:, None]
    slack = tol * rms
    hi = np.abs(y_ref) + slack
    half_place = np.ldexp(1.0, np.frexp(hi)[1] - 9)
    err = np.abs(y - y_ref)
    good = err <= slack + half_place
    assert np.all(good), "bf16 output outside bound at %s" % (np.argwhere(~good)[:5].tolist(),)
    return float(np.max(err / rms))


def unit_k_tiles(in_features, bits):
    """k-tiles per unit of work of the linear's launch (16 where the inputs
    are a multiple of 256 and bits <= 5, else 8)."""
    return 16 if (in_features % 256 == 0 and bits <= 5) else 8


def launch_ctas(num_sms, in_features, out_features, bits):
    """CTAs of one linear launch: one per SM, at most one per unit."""
    units = (out_features // 128) * (in_features // (16 * unit_k_tiles(in_features, bits)))
    return min(units, num_sms)


def cut_blocks(num_sms, in_features, out_features, bits):
    """Output blocks the launch's work split cuts between two or more CTAs
    (their sums go through the cross-CTA partial-sum path): the (block, unit)
    grid, block-major, cut into one contiguous range per CTA."""
    ub = in_features // (16 * unit_k_tiles(in_features, bits))
    units = (out_features // 128) * ub
    ctas = launch_ctas(num_sms, in_features, out_features, bits)
    out = set()
    for c in range(1, ctas):
        u = c * units // ctas          # first unit of CTA c
        if u % ub:
            out.add(u // ub)
    return sorted(out)

"""Comparison of device results with the oracle, with the tolerances of the
hot-path contract:

* fp32 RMS factors: relative error <= 1e-5;
* bf16 outputs: |g - o| <= 1e-3 + 1e-2 |o|;
* block absmax: bit-exact;
* E8M0 scales and element codes, decided in the kernel's precision (the
  oracle's block stage fed the device's own fp32 factors): bit-exact;
* against the oracle's double-precision definition: scales exact except +-1
  where the oracle's normalized absmax lies within 1e-6 (relative) of a
  power-of-two rounding boundary sqrt(2) 2^n (NVFP4: where absmax/6 lies
  within 1e-6 of an E4M3 rounding midpoint); codes exact except one code step
  where the oracle's pre-cast value lies within 1e-6 of a rounding midpoint.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

RINV_RTOL = 1e-5
Y_ATOL, Y_RTOL = 1e-3, 1e-2
NEAR = 1e-6


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits).view(np.int16)
    return torch.from_numpy(b.copy()).view(torch.bfloat16).float().numpy().astype(np.float64)


def check_qk(Y_gpu_bits, rinv_gpu, Y_or_bits, rinv_or, what=""):
    """Returns a dict of statistics; raises AssertionError on a violation."""
    rel = np.abs(rinv_gpu.astype(np.float64) - rinv_or) / np.abs(rinv_or)
    assert rel.max() <= RINV_RTOL, f"{what} rinv rel err {rel.max():.3g}"
    g = bf16_to_f64(Y_gpu_bits)
    o = bf16_to_f64(Y_or_bits)
    bad = np.abs(g - o) > Y_ATOL + Y_RTOL * np.abs(o)
    assert not bad.any(), f"{what} {bad.sum()} bf16 outputs out of tolerance"
    return {"rinv_max_rel": float(rel.max()),
            "y_exact_frac": float(np.mean(Y_gpu_bits == Y_or_bits))}


def _format_values(fmt):
    if fmt == oracle.FMT_E4M3:
        return np.array([oracle.decode(c, fmt) for c in range(0x7F)])
    return np.array([oracle.decode(c, oracle.FMT_E2M1) for c in range(8)])


def _near_midpoint(v, fmt):
    """Relative distance of |v| to the nearest rounding midpoint of fmt."""
    vals = _format_values(fmt)
    mids = (vals[:-1] + vals[1:]) / 2
    return np.min(np.abs(np.abs(v)[:, None] / mids[None, :] - 1), axis=1)


def _near_boundary_log2(v):
    """Relative distance of v > 0 to the nearest sqrt(2) * 2^n."""
    e = np.floor(np.log2(v))
    m = v / np.exp2(e)                      # in [1, 2); the boundary is sqrt(2)
    return np.abs(m / np.sqrt(2) - 1)


def unpack_codes(codes, fmt, D):
    if fmt == oracle.FMT_E4M3:
        return codes
    out = np.empty((codes.shape[0], D), np.uint8)
    out[:, 0::2] = codes & 0xF
    out[:, 1::2] = codes >> 4
    return out


def check_mx(X_bits, gamma, B, fmt, gpu, ref, rinv_gpu, eps, what=""):
    """gpu = (codes, scales, amax or None); ref = oracle outputs
    (codes, scales, rinv f64, amax) of the double-precision definition."""
    codes_g, scales_g, amax_g = gpu
    codes_o, scales_o, rinv_o, amax_o = ref
    T, D = X_bits.shape
    stats = {}
    rel = np.abs(rinv_gpu.astype(np.float64) - rinv_o) / np.abs(rinv_o)
    assert rel.max() <= RINV_RTOL, f"{what} rinv rel err {rel.max():.3g}"
    stats["rinv_max_rel"] = float(rel.max())
    if amax_g is not None:
        assert np.array_equal(amax_g.view(np.uint32), amax_o.view(np.uint32)), f"{what} amax"

    # (1) same-precision decisions: bit-exact
    c_s, s_s, a_s = oracle.mx_cast_given_rinv(X_bits, gamma, rinv_gpu, B, fmt)
    nbad_s = int((scales_g != s_s).sum())
    nbad_c = int((codes_g != c_s).sum())
    assert nbad_s == 0, f"{what} {nbad_s} scales differ from the fp32 block stage"
    assert nbad_c == 0, f"{what} {nbad_c} code bytes differ from the fp32 block stage"

    # (2) against the double definition: exceptions only at boundaries
    nvfp4 = fmt == oracle.FMT_NVFP4
    diff_s = scales_g != scales_o
    stats["scale_boundary_exceptions"] = int(diff_s.sum())
    if diff_s.any():
        v = (amax_o.astype(np.float64) * rinv_o[:, None])[diff_s]
        assert np.all(np.abs(scales_g[diff_s].astype(int) - scales_o[diff_s].astype(int)) == 1)
        near = (_near_midpoint(v / 6.0, oracle.FMT_E4M3) if nvfp4
                else _near_boundary_log2(v))
        assert np.all(near <= NEAR), f"{what} scale differs away from a boundary"
    cg = unpack_codes(codes_g, fmt, D)
    co = unpack_codes(codes_o, fmt, D)
    same_scale = np.repeat(~diff_s, B, axis=1)
    diff_c = (cg != co) & same_scale
    stats["code_boundary_exceptions"] = int(diff_c.sum())
    if diff_c.any():
        vals = _format_values(fmt)
        mids = (vals[:-1] + vals[1:]) / 2
        rows, cols = np.nonzero(diff_c)
        x = bf16_to_f64(X_bits[rows, cols])
        w = x if gamma is None else (x.astype(np.float32) * gamma[cols]).astype(np.float64)
        if nvfp4:
            sc = scales_o[rows, cols // B]
            q = np.abs(w * rinv_o[rows] / np.array([oracle.decode(int(c), oracle.FMT_E4M3)
                                                    for c in sc]))
        else:
            e = scales_o[rows, cols // B].astype(np.float64) - 127
            q = np.abs(w * rinv_o[rows] * np.exp2(-e))
        near = np.min(np.abs(q[:, None] / mids[None, :] - 1), axis=1) <= NEAR
        sign_mask = 0x7F if fmt == oracle.FMT_E4M3 else 0x7
        step = np.abs((cg[rows, cols] & sign_mask).astype(int) - (co[rows, cols] & sign_mask).astype(int))
        assert np.all(near & (step == 1)), f"{what} code differs away from a midpoint"
    return stats

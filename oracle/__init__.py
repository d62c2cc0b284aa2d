"""CPU oracle for the per-token normalization paths -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never does, and this package
imports nothing from the product package.

The arithmetic lives in ``oracle.c`` (plain C, double precision, built with
gcc, no floating-point contraction); this module only marshals numpy arrays
through ctypes.  Each wrapper names the passage its C function follows:

* ``qknorm_rms``       -- SwiftQK, Eq. (1) evaluated in the phases of
                          Algorithm 1 (split-H partial sums, combine, x*gamma,
                          final scaling).
* ``qknorm_rms_fp8``   -- SwiftQK Sec. IV.C: the same on FP8-E4M3 activations.
* ``layernorm_split``  -- SwiftQK notes Sec. 5e: LayerNorm with its two
                          additive statistics split over H.
* ``qknorm_rms_heads`` -- SwiftQK Sec. II.A: headwise QK-Norm, one factor per
                          head, gamma shared by the heads.
* ``rmsnorm_mxcast``   -- MXNorm card, Fig. 1 caption: RMSNorm then MXCast.
* ``mxnorm_cast``      -- MXNorm card, abstract and Fig. 1 caption: RMS
                          estimated from the block absmaxes, c(B, p).
* ``mxnorm_postround_cast`` -- MXNorm card, Fig. A.4 (reading): the estimate
                          from E8M0-rounded absmaxes.
* ``mx_cast_given_rinv`` -- the MX block stage with a given fp32 factor.
* ``mx_correction``    -- c(B, p) by quadrature.

Parity status of every function is recorded in the test files that pin it
(tests/test_oracle_*.py).  Formats: ``fmt`` 0 = E4M3, 1 = E2M1 (both with
E8M0 block scales), 2 = NVFP4 (E2M1 values, B = 16, E4M3 block scales).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_E4M3 = 0
FMT_E2M1 = 1
FMT_NVFP4 = 2


# The mutation tests load a copy of the oracle with a planted mistake from
# the path in this variable (never set outside those tests).
_LIB_OVERRIDE = os.environ.get("NTS_ORACLE_LIB")


def compile_source(src: str, out: str) -> str:
    """gcc src -> shared library `out`, with the flags of the oracle build."""
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fvisibility=hidden", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into oracle/_build/liboracle.so."""
    if _LIB_OVERRIDE:
        return _LIB_OVERRIDE
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_qknorm_rms.argtypes = [P, P, P, P, P, i64, i64, dbl, i32]
        lib.oracle_qknorm_rms_fp8.argtypes = [P, dbl, P, P, P, P, i64, i64, dbl, i32]
        lib.oracle_layernorm_split.argtypes = [P, P, P, P, P, P, P, i64, i64, dbl, i32]
        lib.oracle_qknorm_rms_heads.argtypes = [P, P, P, P, i64, i64, i64, dbl]
        lib.oracle_rmsnorm_mxcast.argtypes = [P, P, P, P, P, P, P, i64, i64, dbl, i32, i32]
        lib.oracle_mxnorm_cast.argtypes = [P, P, P, P, P, P, P, i64, i64, dbl, i32, i32, i32, dbl]
        lib.oracle_mxnorm_postround_cast.argtypes = [P, P, P, P, P, P, P, i64, i64, dbl, i32, i32,
                                                     i32, dbl]
        lib.oracle_mx_cast_given_rinv.argtypes = [P, P, P, P, P, P, P, i64, i64, i32, i32]
        lib.oracle_mx_correction.argtypes = [i32, i32]
        lib.oracle_mx_correction.restype = dbl
        lib.oracle_encode_array.argtypes = [P, P, i64, i32]
        lib.oracle_bf16_array.argtypes = [P, P, i64]
        lib.oracle_e8m0_array.argtypes = [P, P, i64, i32]
        lib.oracle_round_log2.argtypes = [dbl]
        lib.oracle_round_log2.restype = i32
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = dbl
        lib.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_to_double.restype = dbl
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _bf16_bits(X) -> np.ndarray:
    X = np.ascontiguousarray(X)
    if X.dtype != np.uint16:
        raise TypeError("X must hold bfloat16 bit patterns as uint16")
    return X


def _gamma(g, n):
    if g is None:
        return None
    g = np.ascontiguousarray(g, dtype=np.float32)
    if g.shape != (n,):
        raise ValueError("gamma must have shape [H]")
    return g


def codes_row_bytes(D: int, fmt: int) -> int:
    return D if fmt == FMT_E4M3 else D // 2


def qknorm_rms(X, gamma, eps: float, N: int):
    """Returns (Y bf16 bits [T,H], rinv f64 [T], partial sums f64 [T,N])."""
    X = _bf16_bits(X)
    T, H = X.shape
    if N < 1 or H % N:
        raise ValueError("H must be a multiple of N")
    g = _gamma(gamma, H)
    Y = np.empty_like(X)
    rinv = np.empty(T, np.float64)
    part = np.empty((T, N), np.float64)
    _load().oracle_qknorm_rms(_ptr(X), _ptr(g), _ptr(Y), _ptr(rinv), _ptr(part),
                              T, H, float(eps), N)
    return Y, rinv, part


def qknorm_rms_fp8(X_codes, x_scale: float, gamma, eps: float, N: int):
    """QK-RMSNorm of E4M3 activations (value = code * x_scale).
    Returns (Y bf16 bits [T,H], rinv f64 [T], partial sums f64 [T,N])."""
    X = np.ascontiguousarray(X_codes, dtype=np.uint8)
    T, H = X.shape
    if N < 1 or H % N:
        raise ValueError("H must be a multiple of N")
    g = _gamma(gamma, H)
    Y = np.empty((T, H), np.uint16)
    rinv = np.empty(T, np.float64)
    part = np.empty((T, N), np.float64)
    _load().oracle_qknorm_rms_fp8(_ptr(X), float(x_scale), _ptr(g), _ptr(Y), _ptr(rinv),
                                  _ptr(part), T, H, float(eps), N)
    return Y, rinv, part


def layernorm_split(X, gamma, beta, eps: float, N: int):
    """LayerNorm over H split into N shards.  Returns (Y bf16 bits [T,H],
    mean f64 [T], rstd f64 [T], partials f64 [T,N,2] = per-shard (sum x,
    sum x^2))."""
    X = _bf16_bits(X)
    T, H = X.shape
    if N < 1 or H % N:
        raise ValueError("H must be a multiple of N")
    g = _gamma(gamma, H)
    b = _gamma(beta, H)
    Y = np.empty_like(X)
    mean = np.empty(T, np.float64)
    rstd = np.empty(T, np.float64)
    part = np.empty((T, N, 2), np.float64)
    _load().oracle_layernorm_split(_ptr(X), _ptr(g), _ptr(b), _ptr(Y), _ptr(mean), _ptr(rstd),
                                   _ptr(part), T, H, float(eps), N)
    return Y, mean, rstd, part


def qknorm_rms_heads(X, gamma, eps: float, head_dim: int):
    """Headwise QK-Norm: returns (Y bf16 bits [T,H], rinv f64 [T, H/head_dim]);
    gamma has head_dim entries."""
    X = _bf16_bits(X)
    T, H = X.shape
    if head_dim < 1 or H % head_dim:
        raise ValueError("H must be a multiple of head_dim")
    g = _gamma(gamma, head_dim)
    Y = np.empty_like(X)
    rinv = np.empty((T, H // head_dim), np.float64)
    _load().oracle_qknorm_rms_heads(_ptr(X), _ptr(g), _ptr(Y), _ptr(rinv), T, H, head_dim,
                                    float(eps))
    return Y, rinv


def _check_fmt(fmt: int, B: int, post: bool = False):
    if fmt not in (FMT_E4M3, FMT_E2M1, FMT_NVFP4):
        raise ValueError(f"unknown format {fmt}")
    if fmt == FMT_NVFP4 and (B != 16 or post):
        raise ValueError("NVFP4 has 16-value blocks and E4M3 scales (no post-round form)")


def _mx_out(T, D, B, fmt):
    codes = np.empty((T, codes_row_bytes(D, fmt)), np.uint8)
    scales = np.empty((T, D // B), np.uint8)
    amax = np.empty((T, D // B), np.float32)
    return codes, scales, amax


def rmsnorm_mxcast(X, gamma, eps: float, B: int, fmt: int):
    """Returns (codes, scales, rinv f64 [T], amax f32 [T,K])."""
    _check_fmt(fmt, B)
    X = _bf16_bits(X)
    T, D = X.shape
    g = _gamma(gamma, D)
    codes, scales, amax = _mx_out(T, D, B, fmt)
    rinv = np.empty(T, np.float64)
    work = np.empty(D, np.float32)
    _load().oracle_rmsnorm_mxcast(_ptr(X), _ptr(g), _ptr(codes), _ptr(scales),
                                  _ptr(rinv), _ptr(amax), _ptr(work), T, D,
                                  float(eps), B, fmt)
    return codes, scales, rinv, amax


def mxnorm_cast(X, gamma, eps: float, B: int, fmt: int, p: int):
    """Returns (codes, scales, rinv f64 [T], amax f32 [T,K])."""
    _check_fmt(fmt, B)
    X = _bf16_bits(X)
    T, D = X.shape
    g = _gamma(gamma, D)
    codes, scales, amax = _mx_out(T, D, B, fmt)
    rinv = np.empty(T, np.float64)
    work = np.empty(D, np.float32)
    c = mx_correction(B, p)
    _load().oracle_mxnorm_cast(_ptr(X), _ptr(g), _ptr(codes), _ptr(scales),
                               _ptr(rinv), _ptr(amax), _ptr(work), T, D,
                               float(eps), B, fmt, p, c)
    return codes, scales, rinv, amax


def mxnorm_postround_cast(X, gamma, eps: float, B: int, fmt: int, p: int):
    """Post-round MXNorm. Returns (codes, scales, rinv f64 [T], amax f32 [T,K])."""
    _check_fmt(fmt, B, post=True)
    X = _bf16_bits(X)
    T, D = X.shape
    g = _gamma(gamma, D)
    codes, scales, amax = _mx_out(T, D, B, fmt)
    rinv = np.empty(T, np.float64)
    work = np.empty(D, np.float32)
    c = mx_correction(B, p)
    _load().oracle_mxnorm_postround_cast(_ptr(X), _ptr(g), _ptr(codes), _ptr(scales),
                                         _ptr(rinv), _ptr(amax), _ptr(work), T, D,
                                         float(eps), B, fmt, p, c)
    return codes, scales, rinv, amax


def mx_cast_given_rinv(X, gamma, rinv_f32, B: int, fmt: int):
    """Block stage with given fp32 factors. Returns (codes, scales, amax)."""
    _check_fmt(fmt, B)
    X = _bf16_bits(X)
    T, D = X.shape
    g = _gamma(gamma, D)
    r = np.ascontiguousarray(rinv_f32, dtype=np.float32)
    if r.shape != (T,):
        raise ValueError("rinv must have shape [T]")
    codes, scales, amax = _mx_out(T, D, B, fmt)
    work = np.empty(D, np.float32)
    _load().oracle_mx_cast_given_rinv(_ptr(X), _ptr(g), _ptr(r), _ptr(codes),
                                      _ptr(scales), _ptr(amax), _ptr(work), T, D,
                                      B, fmt)
    return codes, scales, amax


_corr_cache: dict = {}


def mx_correction(B: int, p: int) -> float:
    key = (int(B), int(p))
    if key not in _corr_cache:
        _corr_cache[key] = float(_load().oracle_mx_correction(B, p))
    return _corr_cache[key]


def encode(values, fmt: int) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64).ravel()
    out = np.empty(v.shape, np.uint8)
    _load().oracle_encode_array(_ptr(v), _ptr(out), v.size, fmt)
    return out


def to_bf16(values) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64).ravel()
    out = np.empty(v.shape, np.uint16)
    _load().oracle_bf16_array(_ptr(v), _ptr(out), v.size)
    return out


def e8m0_exponent(values, emax: int) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64).ravel()
    out = np.empty(v.shape, np.int32)
    _load().oracle_e8m0_array(_ptr(v), _ptr(out), v.size, emax)
    return out


def round_log2(v: float) -> int:
    return int(_load().oracle_round_log2(float(v)))


def decode(code: int, fmt: int) -> float:
    lib = _load()
    return float(lib.oracle_e4m3_to_double(code) if fmt == FMT_E4M3
                 else lib.oracle_e2m1_to_double(code))

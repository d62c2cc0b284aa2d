"""Torch-facing binding of libnts: argument marshalling only.  Every step of
the computation runs in the library's CUDA kernels; these functions check
tensor placement, allocate missing outputs with torch, and pass raw pointers
and the current CUDA stream through the C ABI.  Names follow the C ABI
(include/nts.h), without the ``nts_`` prefix."""
from __future__ import annotations

import ctypes
from typing import NamedTuple, Optional

import torch

from ._lib import check, lib

FMT_E4M3 = 0
FMT_E2M1 = 1
FMT_NVFP4 = 2   # E2M1 elements, B = 16, E4M3 block scales
_FMT_NAMES = {"e4m3": FMT_E4M3, "e2m1": FMT_E2M1, "nvfp4": FMT_NVFP4,
              FMT_E4M3: FMT_E4M3, FMT_E2M1: FMT_E2M1, FMT_NVFP4: FMT_NVFP4}


class MxOut(NamedTuple):
    codes: torch.Tensor     # uint8 [T, D] (E4M3) or [T, D/2] (E2M1)
    scales: torch.Tensor    # uint8 [T, D/B] E8M0
    rinv: Optional[torch.Tensor]   # fp32 [T]
    amax: Optional[torch.Tensor]   # fp32 [T, D/B]


def _fmt(fmt) -> int:
    try:
        return _FMT_NAMES[fmt.lower() if isinstance(fmt, str) else fmt]
    except KeyError:
        raise ValueError(f"unknown element format {fmt!r}") from None


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(name: str, t: torch.Tensor, dtype) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def codes_row_bytes(D: int, fmt) -> int:
    return D if _fmt(fmt) == FMT_E4M3 else D // 2


def qknorm_rms(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, N: int = 1,
               out: Optional[torch.Tensor] = None, rinv: Optional[torch.Tensor] = None,
               want_rinv: bool = False, stream=None):
    """Layerwise QK-RMSNorm of x [T, H] (bf16) with gain gamma [H] (fp32),
    split into N cluster shards.  Returns (y, rinv or None).  out may be x."""
    _need_cuda("x", x, torch.bfloat16)
    _need_cuda("gamma", gamma, torch.float32)
    T, H = x.shape
    if out is None:
        out = torch.empty_like(x)
    _need_cuda("out", out, torch.bfloat16)
    if rinv is None and want_rinv:
        rinv = torch.empty(T, device=x.device, dtype=torch.float32)
    if rinv is not None:
        _need_cuda("rinv", rinv, torch.float32)
    check(lib().nts_qknorm_rms(_ptr(x), _ptr(gamma), _ptr(out), _ptr(rinv), T, H,
                               float(eps), int(N), _stream(stream)))
    return out, rinv


def qknorm_rms_fp8(x_codes: torch.Tensor, x_scale: float, gamma: torch.Tensor,
                   eps: float = 1e-6, N: int = 1, out: Optional[torch.Tensor] = None,
                   rinv: Optional[torch.Tensor] = None, want_rinv: bool = False, stream=None):
    """QK-RMSNorm of FP8-E4M3 activations: x_codes uint8 (or float8_e4m3fn)
    [T, H], value = code * x_scale.  Returns (y bf16 [T, H], rinv or None)."""
    if x_codes.dtype == torch.float8_e4m3fn:
        x_codes = x_codes.view(torch.uint8)
    _need_cuda("x_codes", x_codes, torch.uint8)
    _need_cuda("gamma", gamma, torch.float32)
    T, H = x_codes.shape
    if out is None:
        out = torch.empty(T, H, device=x_codes.device, dtype=torch.bfloat16)
    _need_cuda("out", out, torch.bfloat16)
    if rinv is None and want_rinv:
        rinv = torch.empty(T, device=x_codes.device, dtype=torch.float32)
    if rinv is not None:
        _need_cuda("rinv", rinv, torch.float32)
    check(lib().nts_qknorm_rms_fp8(_ptr(x_codes), float(x_scale), _ptr(gamma), _ptr(out),
                                   _ptr(rinv), T, H, float(eps), int(N), _stream(stream)))
    return out, rinv


def qknorm_rms_heads(x: torch.Tensor, gamma: torch.Tensor, head_dim: int, eps: float = 1e-6,
                     N: int = 1, out: Optional[torch.Tensor] = None,
                     rinv: Optional[torch.Tensor] = None, want_rinv: bool = False, stream=None):
    """Headwise QK-Norm of x [T, H] (H = nheads * head_dim) with gamma
    [head_dim] shared by the heads.  Returns (y, rinv [T, nheads] or None)."""
    _need_cuda("x", x, torch.bfloat16)
    _need_cuda("gamma", gamma, torch.float32)
    T, H = x.shape
    if out is None:
        out = torch.empty_like(x)
    _need_cuda("out", out, torch.bfloat16)
    if rinv is None and want_rinv:
        rinv = torch.empty(T, H // head_dim, device=x.device, dtype=torch.float32)
    if rinv is not None:
        _need_cuda("rinv", rinv, torch.float32)
    check(lib().nts_qknorm_rms_heads(_ptr(x), _ptr(gamma), _ptr(out), _ptr(rinv), T, H,
                                     int(head_dim), float(eps), int(N), _stream(stream)))
    return out, rinv


def layernorm_split(x: torch.Tensor, gamma: torch.Tensor, beta: Optional[torch.Tensor] = None,
                    eps: float = 1e-5, N: int = 1, out: Optional[torch.Tensor] = None,
                    mean: Optional[torch.Tensor] = None, rstd: Optional[torch.Tensor] = None,
                    want_stats: bool = False, stream=None):
    """LayerNorm of x [T, H] (bf16) with gain gamma and optional shift beta
    (fp32 [H]), the statistics exchanged as per-shard (sum, sum of squares)
    between N cluster shards.  Returns (y, mean or None, rstd or None)."""
    _need_cuda("x", x, torch.bfloat16)
    _need_cuda("gamma", gamma, torch.float32)
    if beta is not None:
        _need_cuda("beta", beta, torch.float32)
    T, H = x.shape
    if out is None:
        out = torch.empty_like(x)
    _need_cuda("out", out, torch.bfloat16)
    if want_stats:
        mean = torch.empty(T, device=x.device, dtype=torch.float32) if mean is None else mean
        rstd = torch.empty(T, device=x.device, dtype=torch.float32) if rstd is None else rstd
    for name, t in (("mean", mean), ("rstd", rstd)):
        if t is not None:
            _need_cuda(name, t, torch.float32)
    check(lib().nts_layernorm_split(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(out), _ptr(mean),
                                    _ptr(rstd), T, H, float(eps), int(N), _stream(stream)))
    return out, mean, rstd


def qknorm_rms_mxcast(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, N: int = 1,
                      B: int = 32, fmt="e4m3", codes=None, scales=None, rinv=None,
                      want_rinv: bool = False, stream=None) -> "MxOut":
    """Layerwise QK-RMSNorm of x [T, H] split into N cluster shards, written
    as an MX / NVFP4 block cast (codes, scales) instead of bf16 rows.
    Returns MxOut(codes, scales, rinv or None, None)."""
    _need_cuda("x", x, torch.bfloat16)
    _need_cuda("gamma", gamma, torch.float32)
    T, H = x.shape
    f = _fmt(fmt)
    codes, scales, rinv, _ = _mx_outputs(x, H, B, f, codes, scales, rinv, None, want_rinv,
                                         False)
    check(lib().nts_qknorm_rms_mxcast(_ptr(x), _ptr(gamma), _ptr(codes), _ptr(scales),
                                      _ptr(rinv), T, H, float(eps), int(N), int(B), f,
                                      _stream(stream)))
    return MxOut(codes, scales, rinv, None)


def qknorm_rms_qk_mxcast(q: torch.Tensor, gamma_q: torch.Tensor, k: torch.Tensor,
                         gamma_k: torch.Tensor, eps: float = 1e-6, N: int = 1, B: int = 32,
                         fmt="e4m3", out_q: Optional["MxOut"] = None,
                         out_k: Optional["MxOut"] = None, want_rinv: bool = False,
                         stream=None):
    """qknorm_rms_mxcast of Q [T, Hq] and K [T, Hk] in one launch.  out_q /
    out_k may carry preallocated (codes, scales, rinv or None) buffers.
    Returns (MxOut for Q, MxOut for K)."""
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("gamma_q", gamma_q, torch.float32), ("gamma_k", gamma_k, torch.float32)):
        _need_cuda(name, t, dt)
    T, Hq = q.shape
    Tk, Hk = k.shape
    if Tk != T:
        raise ValueError("q and k must have the same number of tokens")
    f = _fmt(fmt)
    bufs = []
    for x, H, o in ((q, Hq, out_q), (k, Hk, out_k)):
        c, s_, r = (o.codes, o.scales, o.rinv) if o is not None else (None, None, None)
        c, s_, r, _ = _mx_outputs(x, H, B, f, c, s_, r, None, want_rinv, False)
        bufs.append((c, s_, r))
    (cq, sq, rq), (ck, sk, rk) = bufs
    check(lib().nts_qknorm_rms_qk_mxcast(_ptr(q), _ptr(gamma_q), _ptr(cq), _ptr(sq), _ptr(rq),
                                         _ptr(k), _ptr(gamma_k), _ptr(ck), _ptr(sk), _ptr(rk),
                                         T, Hq, Hk, float(eps), int(N), int(B), f,
                                         _stream(stream)))
    return MxOut(cq, sq, rq, None), MxOut(ck, sk, rk, None)


def qknorm_rms_qk(q: torch.Tensor, gamma_q: torch.Tensor, k: torch.Tensor,
                  gamma_k: torch.Tensor, eps: float = 1e-6, N: int = 1,
                  out_q: Optional[torch.Tensor] = None, out_k: Optional[torch.Tensor] = None,
                  rinv_q: Optional[torch.Tensor] = None, rinv_k: Optional[torch.Tensor] = None,
                  want_rinv: bool = False, stream=None):
    """Layerwise QK-RMSNorm of Q [T, Hq] and K [T, Hk] in one launch.
    Returns (yq, yk, rinv_q or None, rinv_k or None)."""
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("gamma_q", gamma_q, torch.float32), ("gamma_k", gamma_k, torch.float32)):
        _need_cuda(name, t, dt)
    T, Hq = q.shape
    Tk, Hk = k.shape
    if Tk != T:
        raise ValueError("q and k must have the same number of tokens")
    out_q = torch.empty_like(q) if out_q is None else out_q
    out_k = torch.empty_like(k) if out_k is None else out_k
    if want_rinv:
        rinv_q = torch.empty(T, device=q.device, dtype=torch.float32) if rinv_q is None else rinv_q
        rinv_k = torch.empty(T, device=q.device, dtype=torch.float32) if rinv_k is None else rinv_k
    check(lib().nts_qknorm_rms_qk(_ptr(q), _ptr(gamma_q), _ptr(out_q), _ptr(rinv_q), _ptr(k),
                                  _ptr(gamma_k), _ptr(out_k), _ptr(rinv_k), T, Hq, Hk,
                                  float(eps), int(N), _stream(stream)))
    return out_q, out_k, rinv_q, rinv_k


def _mx_outputs(x, D, B, fmt, codes, scales, rinv, amax, want_rinv, want_amax):
    T = x.shape[0]
    if codes is None:
        codes = torch.empty(T, codes_row_bytes(D, fmt), device=x.device, dtype=torch.uint8)
    if scales is None:
        scales = torch.empty(T, D // B, device=x.device, dtype=torch.uint8)
    if rinv is None and want_rinv:
        rinv = torch.empty(T, device=x.device, dtype=torch.float32)
    if amax is None and want_amax:
        amax = torch.empty(T, D // B, device=x.device, dtype=torch.float32)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    if rinv is not None:
        _need_cuda("rinv", rinv, torch.float32)
    if amax is not None:
        _need_cuda("amax", amax, torch.float32)
    return codes, scales, rinv, amax


def rmsnorm_mxcast(x: torch.Tensor, gamma: Optional[torch.Tensor] = None, eps: float = 1e-6,
                   B: int = 32, fmt="e4m3", codes=None, scales=None, rinv=None, amax=None,
                   want_rinv: bool = False, want_amax: bool = False, stream=None) -> MxOut:
    """RMSNorm of x [T, D] fused with the MX cast to E4M3/E2M1 + E8M0 scales."""
    _need_cuda("x", x, torch.bfloat16)
    if gamma is not None:
        _need_cuda("gamma", gamma, torch.float32)
    T, D = x.shape
    f = _fmt(fmt)
    codes, scales, rinv, amax = _mx_outputs(x, D, B, f, codes, scales, rinv, amax,
                                            want_rinv, want_amax)
    check(lib().nts_rmsnorm_mxcast(_ptr(x), _ptr(gamma), _ptr(codes), _ptr(scales), _ptr(rinv),
                                   _ptr(amax), T, D, float(eps), int(B), f, _stream(stream)))
    return MxOut(codes, scales, rinv, amax)


def mxnorm_cast(x: torch.Tensor, gamma: Optional[torch.Tensor] = None, eps: float = 1e-6,
                B: int = 32, fmt="e4m3", p: int = 2, codes=None, scales=None, rinv=None,
                amax=None, want_rinv: bool = False, want_amax: bool = False,
                stream=None) -> MxOut:
    """MXNorm of x [T, D]: RMS estimated from the MX block absmaxes, then the
    MX cast."""
    _need_cuda("x", x, torch.bfloat16)
    if gamma is not None:
        _need_cuda("gamma", gamma, torch.float32)
    T, D = x.shape
    f = _fmt(fmt)
    codes, scales, rinv, amax = _mx_outputs(x, D, B, f, codes, scales, rinv, amax,
                                            want_rinv, want_amax)
    check(lib().nts_mxnorm_cast(_ptr(x), _ptr(gamma), _ptr(codes), _ptr(scales), _ptr(rinv),
                                _ptr(amax), T, D, float(eps), int(B), f, int(p),
                                _stream(stream)))
    return MxOut(codes, scales, rinv, amax)


def mxnorm_postround_cast(x: torch.Tensor, gamma: Optional[torch.Tensor] = None,
                          eps: float = 1e-6, B: int = 32, fmt="e4m3", p: int = 2, codes=None,
                          scales=None, rinv=None, amax=None, want_rinv: bool = False,
                          want_amax: bool = False, stream=None) -> MxOut:
    """Post-round MXNorm: the RMS estimate from E8M0-rounded block absmaxes."""
    _need_cuda("x", x, torch.bfloat16)
    if gamma is not None:
        _need_cuda("gamma", gamma, torch.float32)
    T, D = x.shape
    f = _fmt(fmt)
    codes, scales, rinv, amax = _mx_outputs(x, D, B, f, codes, scales, rinv, amax,
                                            want_rinv, want_amax)
    check(lib().nts_mxnorm_postround_cast(_ptr(x), _ptr(gamma), _ptr(codes), _ptr(scales),
                                          _ptr(rinv), _ptr(amax), T, D, float(eps), int(B), f,
                                          int(p), _stream(stream)))
    return MxOut(codes, scales, rinv, amax)


def mxnorm_correction(B: int, p: int) -> float:
    c = ctypes.c_double()
    check(lib().nts_mxnorm_correction(int(B), int(p), ctypes.byref(c)))
    return c.value


def check_status(stream=None) -> None:
    """Synchronize the stream and raise if a kernel timed out or failed."""
    check(lib().nts_check_status(_stream(stream)))


# ----------------------------------------------------------- host-buffer forms

def _need_host(name: str, t: torch.Tensor) -> None:
    if t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host tensor")


def qknorm_rms_host(x_host, gamma_dev, y_host, x_dev, y_dev, eps=1e-6, N=1, rinv_host=None,
                    rinv_dev=None, stream=None) -> None:
    """Enqueue H2D copy of x, the kernel, and D2H copies of y (and rinv)."""
    _need_host("x_host", x_host)
    _need_host("y_host", y_host)
    T, H = x_host.shape
    check(lib().nts_qknorm_rms_host(_ptr(x_host), _ptr(gamma_dev), _ptr(y_host), _ptr(rinv_host),
                                    _ptr(x_dev), _ptr(y_dev), _ptr(rinv_dev), T, H, float(eps),
                                    int(N), _stream(stream)))


def qknorm_rms_qk_host(q_host, gamma_q_dev, yq_host, k_host, gamma_k_dev, yk_host, q_dev,
                       yq_dev, k_dev, yk_dev, eps=1e-6, N=1, stream=None) -> None:
    """Enqueue the H2D copies of q and k, the one launch normalizing both,
    and the D2H copies of yq and yk."""
    for name, t in (("q_host", q_host), ("yq_host", yq_host), ("k_host", k_host),
                    ("yk_host", yk_host)):
        _need_host(name, t)
    T, Hq = q_host.shape
    Tk, Hk = k_host.shape
    if Tk != T:
        raise ValueError("q and k must have the same number of tokens")
    check(lib().nts_qknorm_rms_qk_host(
        _ptr(q_host), _ptr(gamma_q_dev), _ptr(yq_host), _ptr(k_host), _ptr(gamma_k_dev),
        _ptr(yk_host), _ptr(q_dev), _ptr(yq_dev), _ptr(k_dev), _ptr(yk_dev), T, Hq, Hk,
        float(eps), int(N), _stream(stream)))


def rmsnorm_mxcast_host(x_host, gamma_dev, codes_host, scales_host, x_dev, codes_dev,
                        scales_dev, eps=1e-6, B=32, fmt="e4m3", stream=None) -> None:
    _need_host("x_host", x_host)
    T, D = x_host.shape
    check(lib().nts_rmsnorm_mxcast_host(_ptr(x_host), _ptr(gamma_dev), _ptr(codes_host),
                                        _ptr(scales_host), _ptr(x_dev), _ptr(codes_dev),
                                        _ptr(scales_dev), T, D, float(eps), int(B), _fmt(fmt),
                                        _stream(stream)))


def mxnorm_cast_host(x_host, gamma_dev, codes_host, scales_host, x_dev, codes_dev, scales_dev,
                     eps=1e-6, B=32, fmt="e4m3", p=2, stream=None) -> None:
    _need_host("x_host", x_host)
    T, D = x_host.shape
    check(lib().nts_mxnorm_cast_host(_ptr(x_host), _ptr(gamma_dev), _ptr(codes_host),
                                     _ptr(scales_host), _ptr(x_dev), _ptr(codes_dev),
                                     _ptr(scales_dev), T, D, float(eps), int(B), _fmt(fmt),
                                     int(p), _stream(stream)))


# ------------------------------------------------------------------ tuning

def mxnorm_cast_host_noalloc(x_host, gamma_host, codes_host, scales_host, eps=1e-6, B=32,
                             fmt="e4m3", p=2, stream=None) -> None:
    """MXNorm of host rows with the library's fixed device staging (no
    caller-owned device buffers; calls that overlap in time race)."""
    _need_host("x_host", x_host)
    T, D = x_host.shape
    if gamma_host is not None:
        _need_host("gamma_host", gamma_host)
    check(lib().nts_mxnorm_cast_host_noalloc(_ptr(x_host), _ptr(gamma_host), _ptr(codes_host),
                                             _ptr(scales_host), T, D, float(eps), int(B),
                                             _fmt(fmt), int(p), _stream(stream)))


def set_tuning(vpt=0, rows=0, stages=0, grid=0, smem_budget=0) -> None:
    check(lib().nts_debug_set_tuning(int(vpt), int(rows), int(stages), int(grid),
                                     int(smem_budget)))


def set_wait_limit_ns(ns: int) -> None:
    check(lib().nts_debug_set_wait_limit_ns(int(ns)))


def set_schedule(dynamic: bool) -> None:
    check(lib().nts_debug_set_schedule(1 if dynamic else 0))


def set_direct(on: bool) -> None:
    check(lib().nts_debug_set_direct(1 if on else 0))


def check_nvfp4_scale() -> tuple:
    """(code mismatches, quotient mismatches) of the kernels' NVFP4 block
    scale against the IEEE-division route over every non-negative fp32
    absmax (nts_debug_check_nvfp4_scale); runs on the current device."""
    a, b = ctypes.c_uint64(0), ctypes.c_uint64(0)
    check(lib().nts_debug_check_nvfp4_scale(ctypes.byref(a), ctypes.byref(b)))
    return int(a.value), int(b.value)


def set_host_chunks(max_chunks: int = 0, min_chunk_bytes: int = 0) -> None:
    """Chunking of the host-buffer forms (0, 0 = defaults); results do not
    depend on it (nts_debug_set_host_chunks)."""
    check(lib().nts_debug_set_host_chunks(int(max_chunks), int(min_chunk_bytes)))


def inject_failure(status: str = "CUDA", count: int = 1) -> None:
    """The next `count` launches fail with NTS_ERR_<status> (CUDA,
    UNSUPPORTED or TIMEOUT) without touching the device; count=0 turns the
    hook off (nts_debug_inject_failure)."""
    codes = {"CUDA": 3, "UNSUPPORTED": 2, "TIMEOUT": 4}
    check(lib().nts_debug_inject_failure(codes[status], int(count)))


def set_pdl(on: bool) -> None:
    """Launch with programmatic stream serialization (default on); results
    do not depend on it (nts_debug_set_pdl)."""
    check(lib().nts_debug_set_pdl(1 if on else 0))


def check_e8m0() -> int:
    """Absmaxes whose E8M0 exponent, as the kernels form it, differs from
    the field-by-field definition (nts_debug_check_e8m0); 0 when right."""
    a = ctypes.c_uint64(0)
    check(lib().nts_debug_check_e8m0(ctypes.byref(a)))
    return int(a.value)


def set_missing_tx(nbytes: int) -> None:
    check(lib().nts_debug_set_missing_tx(int(nbytes)))

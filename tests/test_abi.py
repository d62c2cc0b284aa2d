"""The C ABI without a GPU: the library loads, exports every function the
public headers declare (and no other nts_ symbol), and rejects bad arguments
before touching the device.  Also checks the library's host-side c(B, p)
against the oracle's independent quadrature."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import oracle
from conftest import ROOT

nts = pytest.importorskip("normalization_token_split_gb300")
from normalization_token_split_gb300 import _lib  # noqa: E402

INVALID, UNSUPPORTED, OK = 1, 2, 0
P = ctypes.c_void_p
A16 = P(1 << 20)          # a 16-byte aligned non-NULL address; never dereferenced
MIS = P((1 << 20) + 4)    # misaligned


def header_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(nts_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    return _lib.lib()


def test_every_declared_symbol_is_exported(lib):
    fns = header_functions()
    assert len(fns) >= 14
    for name in fns:
        assert hasattr(lib, name), name


def test_no_undeclared_exports():
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b(nts_\w+)$", out, flags=re.M))
    assert exported == set(header_functions())


def test_status_strings_and_version(lib):
    assert lib.nts_version() >= 100
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.nts_status_string(code).decode() == name


def _qk(lib, X=A16, g=A16, Y=A16, r=None, T=4, H=64, eps=1e-6, N=2):
    return lib.nts_qknorm_rms(X, g, Y, r, T, H, eps, N, None)


def test_qknorm_argument_checks(lib):
    assert _qk(lib, X=None) == INVALID
    assert _qk(lib, g=None) == INVALID
    assert _qk(lib, Y=None) == INVALID
    assert _qk(lib, T=-1) == INVALID
    assert _qk(lib, H=0) == INVALID
    assert _qk(lib, N=3) == INVALID
    assert _qk(lib, H=66, N=4) == INVALID
    assert _qk(lib, eps=0.0) == INVALID
    assert _qk(lib, eps=float("nan")) == INVALID
    assert _qk(lib, eps=float("inf")) == INVALID
    assert _qk(lib, H=8, N=2) == UNSUPPORTED           # H/N = 4 is not a multiple of 8
    assert _qk(lib, H=30728 * 2, N=2) == UNSUPPORTED   # shard wider than 30720
    assert _qk(lib, X=MIS) == UNSUPPORTED
    assert _qk(lib, Y=MIS) == UNSUPPORTED
    assert _qk(lib, T=0) == OK                           # nothing launched
    assert _qk(lib, T=0, X=None, g=None, Y=None) == OK  # empty tensors
    assert _qk(lib, T=0, N=3) == INVALID


def _mx(lib, fn, X=A16, codes=A16, scales=A16, T=4, D=256, eps=1e-6, B=32, fmt=0, p=2):
    if fn == "rms":
        return lib.nts_rmsnorm_mxcast(X, None, codes, scales, None, None, T, D, eps, B, fmt, None)
    return lib.nts_mxnorm_cast(X, None, codes, scales, None, None, T, D, eps, B, fmt, p, None)


@pytest.mark.parametrize("fn", ["rms", "mx"])
def test_mx_argument_checks(lib, fn):
    assert _mx(lib, fn, X=None) == INVALID
    assert _mx(lib, fn, codes=None) == INVALID
    assert _mx(lib, fn, scales=None) == INVALID
    assert _mx(lib, fn, T=-1) == INVALID
    assert _mx(lib, fn, D=0) == INVALID
    assert _mx(lib, fn, B=8) == INVALID
    assert _mx(lib, fn, D=48, B=32) == INVALID
    assert _mx(lib, fn, fmt=2) == INVALID
    assert _mx(lib, fn, eps=-1.0) == INVALID
    if fn == "mx":
        assert _mx(lib, fn, p=3) == INVALID
    assert _mx(lib, fn, D=65536) == UNSUPPORTED
    assert _mx(lib, fn, X=MIS) == UNSUPPORTED
    assert _mx(lib, fn, T=0) == OK
    assert _mx(lib, fn, T=0, X=None, codes=None, scales=None) == OK
    assert _mx(lib, fn, T=0, B=8) == INVALID
    assert len(lib.nts_last_error()) > 0


def test_host_forms_argument_checks(lib):
    assert lib.nts_qknorm_rms_host(None, A16, A16, None, A16, A16, None, 4, 64, 1e-6, 2,
                                   None) == INVALID
    assert lib.nts_qknorm_rms_host(A16, A16, A16, A16, A16, A16, None, 4, 64, 1e-6, 2,
                                   None) == INVALID            # rinv_host without staging
    assert lib.nts_mxnorm_cast_host(A16, None, A16, None, A16, A16, A16, 4, 256, 1e-6, 32, 0, 2,
                                    None) == INVALID
    assert lib.nts_rmsnorm_mxcast_host(A16, None, A16, A16, A16, A16, A16, 0, 256, 1e-6, 32, 0,
                                       None) == OK


def test_fused_qk_host_form_argument_checks(lib):
    def f(**k):
        return lib.nts_qknorm_rms_qk_host(
            k.get("Q", A16), A16, k.get("Yq", A16), k.get("K", A16), A16, A16, A16, A16,
            k.get("Kd", A16), A16, k.get("T", 4), 64, k.get("Hk", 64), 1e-6, k.get("N", 2), None)
    assert f(Q=None) == INVALID
    assert f(Yq=None) == INVALID
    assert f(K=None) == INVALID
    assert f(Hk=65) == INVALID
    assert f(N=3) == INVALID
    assert f(Kd=MIS) == UNSUPPORTED
    assert f(T=0, Q=None, K=None, Yq=None) == OK


def test_debug_hooks_validate(lib):
    assert lib.nts_debug_set_tuning(9, 0, 0, 0, 0) == INVALID
    assert lib.nts_debug_set_tuning(-1, 0, 0, 0, 0) == INVALID
    assert lib.nts_debug_set_missing_tx(17) == INVALID
    assert lib.nts_debug_check_nvfp4_scale(None, None) == INVALID
    assert lib.nts_debug_check_e8m0(None) == INVALID
    assert lib.nts_debug_set_pdl(2) == INVALID
    assert lib.nts_debug_set_pdl(1) == OK
    assert lib.nts_debug_set_host_chunks(65, 0) == INVALID
    assert lib.nts_debug_set_host_chunks(-1, 0) == INVALID
    assert lib.nts_debug_set_host_chunks(0, 0) == OK
    assert lib.nts_debug_set_tuning(0, 0, 0, 0, 0) == OK
    assert lib.nts_debug_set_missing_tx(0) == OK
    assert lib.nts_debug_set_wait_limit_ns(0) == OK


@pytest.mark.parametrize("B", [1, 2, 16, 32, 64])
@pytest.mark.parametrize("p", [1, 2])
def test_library_correction_matches_oracle(B, p):
    assert nts.mxnorm_correction(B, p) == pytest.approx(oracle.mx_correction(B, p), rel=1e-10)


def test_correction_rejects_bad_args(lib):
    c = ctypes.c_double()
    assert lib.nts_mxnorm_correction(0, 2, ctypes.byref(c)) == INVALID
    assert lib.nts_mxnorm_correction(32, 3, ctypes.byref(c)) == INVALID
    assert lib.nts_mxnorm_correction(32, 2, None) == INVALID


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()


def test_headwise_argument_checks(lib):
    f = lambda **k: lib.nts_qknorm_rms_heads(k.get("X", A16), A16, A16, None, k.get("T", 4),
                                             k.get("H", 512), k.get("hd", 128), 1e-6,
                                             k.get("N", 1), None)
    assert f(hd=0) == INVALID
    assert f(H=500) == INVALID
    assert f(T=-1) == INVALID
    assert f(X=None) == INVALID
    assert f(N=3) == INVALID
    assert f(hd=32, H=512, N=8) == UNSUPPORTED       # 4-value shards
    assert f(T=0, X=None) == OK


def test_fp8_argument_checks(lib):
    f = lambda **k: lib.nts_qknorm_rms_fp8(k.get("X", A16), k.get("s", 1.0), A16, A16, None,
                                           k.get("T", 4), k.get("H", 512), 1e-6, k.get("N", 2),
                                           None)
    assert f(s=0.0) == INVALID
    assert f(s=float("nan")) == INVALID
    assert f(X=None) == INVALID
    assert f(H=24, N=1) == UNSUPPORTED          # 24-byte E4M3 rows
    assert f(H=48, N=2) == UNSUPPORTED
    assert f(T=0, X=None) == OK


def test_layernorm_argument_checks(lib):
    def f(**k):
        return lib.nts_layernorm_split(k.get("X", A16), k.get("g", A16), k.get("b", None), A16,
                                       k.get("m", None), None, k.get("T", 4), k.get("H", 512),
                                       k.get("eps", 1e-5), k.get("N", 2), None)
    assert f(X=None) == INVALID
    assert f(g=None) == INVALID
    assert f(T=-1) == INVALID
    assert f(N=3) == INVALID
    assert f(eps=0.0) == INVALID
    assert f(H=8, N=2) == UNSUPPORTED               # 4-value shards
    assert f(b=MIS) == UNSUPPORTED
    assert f(m=P((1 << 20) + 2)) == UNSUPPORTED
    assert f(b=A16, H=20488 * 2, N=2) == UNSUPPORTED  # gamma and beta do not fit on chip
    assert f(T=0, X=None, g=None) == OK


def test_nvfp4_argument_checks(lib):
    NV = 2
    assert lib.nts_rmsnorm_mxcast(A16, None, A16, A16, None, None, 4, 256, 1e-6, 32, NV,
                                  None) == INVALID
    assert lib.nts_mxnorm_cast(A16, None, A16, A16, None, None, 4, 256, 1e-6, 64, NV, 2,
                               None) == INVALID
    assert lib.nts_mxnorm_postround_cast(A16, None, A16, A16, None, None, 4, 256, 1e-6, 16, NV,
                                         2, None) == INVALID
    assert lib.nts_rmsnorm_mxcast(A16, None, A16, A16, None, None, 4, 256, 1e-6, 16, 3,
                                  None) == INVALID
    assert lib.nts_rmsnorm_mxcast(A16, None, A16, A16, None, None, 0, 256, 1e-6, 16, NV,
                                  None) == OK


def test_qk_mxcast_argument_checks(lib):
    def f(**k):
        return lib.nts_qknorm_rms_mxcast(k.get("X", A16), A16, k.get("c", A16), k.get("s", A16),
                                         None, k.get("T", 4), k.get("H", 1024), 1e-6,
                                         k.get("N", 2), k.get("B", 32), k.get("fmt", 0), None)
    assert f(s=None) == INVALID
    assert f(c=None) == INVALID
    assert f(B=8) == INVALID
    assert f(fmt=3) == INVALID
    assert f(fmt=2, B=32) == INVALID
    assert f(H=1040, B=16) == UNSUPPORTED      # 520-value shards
    assert f(c=MIS) == UNSUPPORTED
    assert f(T=0, X=None, c=None, s=None) == OK


def test_injected_launch_failures_reach_the_caller(lib):
    CUDA, TIMEOUT = 3, 4
    try:
        assert lib.nts_debug_inject_failure(CUDA, 2) == OK
        assert _qk(lib) == CUDA                       # arguments pass; the launch "fails"
        assert b"injected" in lib.nts_last_error()
        assert _mx(lib, "mx") == CUDA
        assert lib.nts_debug_inject_failure(TIMEOUT, 1) == OK
        assert _qk(lib) == TIMEOUT
        assert _qk(lib, H=7) == INVALID               # argument checks still come first
        assert lib.nts_debug_inject_failure(1, 1) == INVALID
        assert lib.nts_debug_inject_failure(CUDA, -1) == INVALID
    finally:
        assert lib.nts_debug_inject_failure(0, 0) == OK


def test_qk_mxcast_fused_argument_checks(lib):
    def f(**k):
        return lib.nts_qknorm_rms_qk_mxcast(
            k.get("Q", A16), A16, k.get("cq", A16), k.get("sq", A16), None,
            k.get("K", A16), A16, k.get("ck", A16), k.get("sk", A16), None,
            k.get("T", 4), k.get("Hq", 1024), k.get("Hk", 512), 1e-6, k.get("N", 2),
            k.get("B", 32), k.get("fmt", 0), None)
    assert f(sq=None) == INVALID
    assert f(sk=None) == INVALID
    assert f(K=None) == INVALID
    assert f(B=8) == INVALID
    assert f(fmt=2, B=32) == INVALID
    assert f(Hk=1040, B=16) == UNSUPPORTED     # K shards of 520 values
    assert f(ck=MIS) == UNSUPPORTED
    assert f(T=0, Q=None, K=None, cq=None, sq=None, ck=None, sk=None) == OK


def test_noalloc_argument_checks(lib):
    f = lambda **k: lib.nts_mxnorm_cast_host_noalloc(
        k.get("X", A16), k.get("g", None), A16, A16, k.get("T", 4), k.get("D", 256),
        k.get("eps", 1e-6), k.get("B", 32), k.get("fmt", 0), k.get("p", 2), None)
    assert f(X=None) == INVALID
    assert f(B=8) == INVALID
    assert f(p=3) == INVALID
    assert f(fmt=5) == INVALID
    assert f(T=-1) == INVALID
    assert f(T=4096, D=4096) == UNSUPPORTED      # beyond the 16 MiB static scratch
    assert b"static scratch" in lib.nts_last_error()
    assert f(T=0, X=None) == OK
    # sizes whose byte counts would wrap around 64 bits are refused before
    # any product is formed
    assert f(T=1 << 53, D=32768, B=16) == UNSUPPORTED
    assert f(T=(1 << 63) - 1, D=32768, B=64, fmt=1) == UNSUPPORTED
    assert f(T=4, D=65536) == UNSUPPORTED
    # a refused call enqueues nothing, not even the gamma copy (with no GPU
    # here, an enqueued copy would surface as a CUDA error, not INVALID)
    assert f(g=A16, eps=0.0) == INVALID
    assert f(g=A16, fmt=2, B=32) == INVALID      # NVFP4 blocks are 16 values
    assert f(g=A16, B=24, D=240) == INVALID

"""ctypes loader of the in-tree libnts.so.  There is no fallback: if the
library has not been built (``normalization_token_split_gb300.build``) every
call raises."""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libnts.so")

_lock = threading.Lock()
_lib = None

NTS_OK = 0
STATUS_NAMES = {0: "NTS_OK", 1: "NTS_ERR_INVALID_ARG", 2: "NTS_ERR_UNSUPPORTED",
                3: "NTS_ERR_CUDA", 4: "NTS_ERR_TIMEOUT"}


class NtsError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")


def _declare(lib):
    P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    sig = {
        "nts_version": ([], i32),
        "nts_status_string": ([i32], ctypes.c_char_p),
        "nts_last_error": ([], ctypes.c_char_p),
        "nts_qknorm_rms": ([P, P, P, P, i64, i64, f32, i32, P], i32),
        "nts_qknorm_rms_qk": ([P, P, P, P, P, P, P, P, i64, i64, i64, f32, i32, P], i32),
        "nts_layernorm_split": ([P, P, P, P, P, P, i64, i64, f32, i32, P], i32),
        "nts_qknorm_rms_mxcast": ([P, P, P, P, P, i64, i64, f32, i32, i32, i32, P], i32),
        "nts_qknorm_rms_qk_mxcast": ([P, P, P, P, P, P, P, P, P, P, i64, i64, i64, f32, i32, i32,
                                      i32, P], i32),
        "nts_qknorm_rms_fp8": ([P, f32, P, P, P, i64, i64, f32, i32, P], i32),
        "nts_qknorm_rms_heads": ([P, P, P, P, i64, i64, i64, f32, i32, P], i32),
        "nts_rmsnorm_mxcast": ([P, P, P, P, P, P, i64, i64, f32, i32, i32, P], i32),
        "nts_mxnorm_cast": ([P, P, P, P, P, P, i64, i64, f32, i32, i32, i32, P], i32),
        "nts_mxnorm_postround_cast": ([P, P, P, P, P, P, i64, i64, f32, i32, i32, i32, P], i32),
        "nts_mxnorm_correction": ([i32, i32, ctypes.POINTER(ctypes.c_double)], i32),
        "nts_check_status": ([P], i32),
        "nts_qknorm_rms_host": ([P, P, P, P, P, P, P, i64, i64, f32, i32, P], i32),
        "nts_rmsnorm_mxcast_host": ([P, P, P, P, P, P, P, i64, i64, f32, i32, i32, P], i32),
        "nts_mxnorm_cast_host": ([P, P, P, P, P, P, P, i64, i64, f32, i32, i32, i32, P], i32),
        "nts_qknorm_rms_qk_host": ([P, P, P, P, P, P, P, P, P, P, i64, i64, i64, f32, i32, P],
                                   i32),
        "nts_mxnorm_cast_host_noalloc": ([P, P, P, P, i64, i64, f32, i32, i32, i32, P], i32),
        "nts_debug_set_tuning": ([i32, i32, i32, i64, i32], i32),
        "nts_debug_set_wait_limit_ns": ([ctypes.c_uint64], i32),
        "nts_debug_set_missing_tx": ([ctypes.c_uint32], i32),
        "nts_debug_set_schedule": ([i32], i32),
        "nts_debug_set_direct": ([i32], i32),
        "nts_debug_set_pdl": ([i32], i32),
        "nts_debug_mx_launch_shape": ([i64, i64, i32, i32, i32, i32, i32, i32,
                                       ctypes.POINTER(ctypes.c_int32)], i32),
        "nts_debug_inject_failure": ([i32, i32], i32),
        "nts_debug_check_e8m0": ([ctypes.POINTER(ctypes.c_uint64)], i32),
        "nts_debug_set_host_chunks": ([i32, i64], i32),
        "nts_debug_check_nvfp4_scale": ([ctypes.POINTER(ctypes.c_uint64),
                                         ctypes.POINTER(ctypes.c_uint64)], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res


def lib():
    """The loaded library; raises if it was never built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libnts.so is not built ({LIB_PATH} missing); run "
                    "`python -m normalization_token_split_gb300.build`")
            handle = ctypes.CDLL(LIB_PATH)
            _declare(handle)
            _lib = handle
        return _lib


def check(status: int) -> None:
    if status != NTS_OK:
        detail = lib().nts_last_error().decode(errors="replace")
        raise NtsError(status, detail)

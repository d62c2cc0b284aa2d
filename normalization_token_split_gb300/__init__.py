"""GB300-native per-token RMS normalization.

Two hot paths, both hand-written sm_103a CUDA behind a C ABI (include/nts.h):

* ``qknorm_rms``      layerwise QK-RMSNorm with split-H scalar partial sums,
                      the shards mapped onto the CTAs of a thread-block cluster
                      (SwiftQK, Eq. (1) and Algorithm 1);
* ``rmsnorm_mxcast``  RMSNorm fused with the MX block cast (E4M3 / E2M1 values,
                      E8M0 scales);
* ``mxnorm_cast``     MXNorm: the RMS estimated from the MX block absmaxes,
                      fused with the same cast (MXNorm card, Fig. 1).

Build the library with ``python -m normalization_token_split_gb300.build``.
"""
from ._lib import NtsError
from .ops import (FMT_E2M1, FMT_E4M3, FMT_NVFP4, MxOut, check_status, codes_row_bytes, mxnorm_cast,
                  mxnorm_cast_host, mxnorm_cast_host_noalloc, mxnorm_correction, mxnorm_postround_cast, qknorm_rms, qknorm_rms_host, qknorm_rms_qk_host,
                  qknorm_rms_fp8, qknorm_rms_heads, qknorm_rms_qk, layernorm_split, qknorm_rms_mxcast,
                  qknorm_rms_qk_mxcast,
                  rmsnorm_mxcast, rmsnorm_mxcast_host, set_missing_tx, set_schedule, set_direct, set_tuning,
                  set_wait_limit_ns, check_nvfp4_scale, set_pdl, set_host_chunks,
                  check_e8m0, inject_failure)

__all__ = [
    "NtsError", "FMT_E4M3", "FMT_E2M1", "FMT_NVFP4", "MxOut", "qknorm_rms", "qknorm_rms_fp8", "qknorm_rms_heads", "qknorm_rms_qk", "layernorm_split", "qknorm_rms_mxcast", "qknorm_rms_qk_mxcast", "rmsnorm_mxcast", "mxnorm_cast", "mxnorm_postround_cast",
    "mxnorm_correction", "check_status", "codes_row_bytes", "qknorm_rms_host", "qknorm_rms_qk_host",
    "rmsnorm_mxcast_host", "mxnorm_cast_host", "mxnorm_cast_host_noalloc", "set_tuning", "set_wait_limit_ns",
    "set_missing_tx", "set_schedule", "set_direct", "check_nvfp4_scale", "set_pdl", "set_host_chunks", "check_e8m0", "inject_failure",
]

"""GPU parity of nts_qknorm_rms_mxcast (split-H QK-RMSNorm whose rows leave
as an MX / NVFP4 block cast) against the oracle, through the C ABI.

The oracle is the RMSNorm + block cast definition (oracle.rmsnorm_mxcast with
the gain): N changes only the fp32 summation order of the statistic.  Scales
and codes are compared bit-exactly with the oracle's block stage fed the
device's own fp32 factors, and against the double-precision definition with
exceptions only at rounding boundaries (tests/parity.py)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_mx

pytestmark = pytest.mark.gpu

nts = pytest.importorskip("normalization_token_split_gb300")
DEV = "cuda:0"
FMTS = {"e4m3": oracle.FMT_E4M3, "e2m1": oracle.FMT_E2M1, "nvfp4": oracle.FMT_NVFP4}
FB = [("e4m3", 16), ("e4m3", 32), ("e4m3", 64), ("e2m1", 32), ("e2m1", 64), ("nvfp4", 16)]


def run_and_check(X, g, N, fmt, B, rows=None, eps=1e-6, what=""):
    out = nts.qknorm_rms_mxcast(X.to(DEV), g.to(DEV), eps=eps, N=N, B=B, fmt=fmt,
                                want_rinv=True)
    nts.check_status()
    sel = slice(None) if rows is None else rows
    codes = out.codes[sel].cpu().numpy()
    scales = out.scales[sel].cpu().numpy()
    rinv = out.rinv[sel].cpu().numpy()
    Xb = workloads.bf16_bits(X[sel])
    gn = g.cpu().numpy()
    ref = oracle.rmsnorm_mxcast(Xb, gn, eps, B, FMTS[fmt])
    return check_mx(Xb, gn, B, FMTS[fmt], (codes, scales, None), ref, rinv, eps, what), out


@pytest.mark.parametrize("fmt,B", FB)
@pytest.mark.parametrize("N", [1, 2, 4, 8])
@pytest.mark.parametrize("T,H", [(1, 4096), (37, 5120), (513, 1024), (64, 2048)])
def test_matches_oracle(fmt, B, N, T, H):
    X, g = workloads.qk_inputs(T, H, seed=T + H + N, outlier_frac=0.01)
    run_and_check(X, g, N, fmt, B, what=f"{fmt} B={B} N={N} T={T} H={H}")


@pytest.mark.parametrize("fmt,B", [("e4m3", 32), ("nvfp4", 16), ("e2m1", 32)])
def test_prefill_full_size_sampled(fmt, B):
    X, g = workloads.qk_inputs(8192, 5120, seed=3000, outlier_frac=0.01, device=DEV)
    rng = np.random.default_rng(7)
    rows = torch.from_numpy(np.unique(np.concatenate([rng.choice(8192, 512, replace=False),
                                                      [0, 8191]]))).to(DEV)
    run_and_check(X, g, 4, fmt, B, rows=rows, what=f"prefill {fmt}")


def test_rinv_equals_the_bf16_output_kernel():
    # same statistic, same summation order: the factors are bit-identical
    X, g = workloads.qk_inputs(1000, 4096, seed=55, device=DEV)
    for N in (1, 4):
        out = nts.qknorm_rms_mxcast(X, g, N=N, B=32, fmt="e4m3", want_rinv=True)
        _, r = nts.qknorm_rms(X, g, N=N, want_rinv=True)
        nts.check_status()
        assert torch.equal(out.rinv, r)


def test_degenerate_rows():
    X, g = workloads.qk_inputs(40, 2048, seed=56)
    X[0] = 0
    X[1, :64] = 0
    X[2, 100:140] = 3.0e4
    for fmt, B in (("e4m3", 32), ("nvfp4", 16), ("e2m1", 64)):
        run_and_check(X, g, 2, fmt, B, what=f"degenerate {fmt}")


def test_zero_tokens_and_unsplittable_blocks():
    E = torch.empty(0, 1024, dtype=torch.bfloat16, device=DEV)
    g = torch.ones(1024, device=DEV)
    out = nts.qknorm_rms_mxcast(E, g, N=2, B=32)
    nts.check_status()
    assert out.codes.shape == (0, 1024)
    # shards of 520 values cannot hold whole 16-value blocks
    X = torch.ones(4, 1040, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nts.NtsError, match="UNSUPPORTED"):
        nts.qknorm_rms_mxcast(X, torch.ones(1040, device=DEV), N=2, B=16, fmt="e4m3")


@pytest.mark.parametrize("vpt,rows,stages,grid", [(1, 1, 1, 1), (2, 3, 2, 5), (8, 2, 4, 0)])
def test_forced_launch_shapes(vpt, rows, stages, grid):
    X, g = workloads.qk_inputs(777, 2048, seed=57)
    try:
        nts.set_tuning(vpt=vpt, rows=rows, stages=stages, grid=grid)
        for N in (1, 4):
            run_and_check(X, g, N, "e4m3", 32, what=f"forced {vpt},{rows},{stages},{grid}")
    finally:
        nts.set_tuning()

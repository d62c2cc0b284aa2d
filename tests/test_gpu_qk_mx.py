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


# ------------------------------------------- Q and K in one launch (f1 + f4)

@pytest.mark.parametrize("fmt,B", [("e4m3", 32), ("e2m1", 64), ("nvfp4", 16), ("e4m3", 16)])
@pytest.mark.parametrize("N", [1, 2, 4])
@pytest.mark.parametrize("T,Hq,Hk", [(1, 4096, 1024), (37, 5120, 5120), (300, 2048, 512),
                                     (2000, 4096, 4096)])
def test_fused_q_and_k(fmt, B, N, T, Hq, Hk):
    # Both tensors share the row shape of the wider shard, so with equal
    # widths each tensor's arithmetic and summation order are those of a
    # one-tensor call (bit for bit); with unequal widths the narrower one
    # sums in another order: rinv within fp32 rounding, and the scales and
    # codes those the oracle's block stage gives for the device's rinv.
    Q, gq = workloads.qk_inputs(T, Hq, seed=T + Hq + N, outlier_frac=0.01, device=DEV)
    K, gk = workloads.qk_inputs(T, Hk, seed=T + Hk + N + 1, device=DEV)
    oq, ok = nts.qknorm_rms_qk_mxcast(Q, gq, K, gk, N=N, B=B, fmt=fmt, want_rinv=True)
    sq = nts.qknorm_rms_mxcast(Q, gq, N=N, B=B, fmt=fmt, want_rinv=True)
    sk = nts.qknorm_rms_mxcast(K, gk, N=N, B=B, fmt=fmt, want_rinv=True)
    nts.check_status()
    for X, g, a, b, tag in ((Q, gq, oq, sq, "Q"), (K, gk, ok, sk, "K")):
        if Hq == Hk:
            assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
            assert torch.equal(a.rinv, b.rinv)
            continue
        assert torch.max(torch.abs(a.rinv / b.rinv - 1)).item() < 1e-6
        Xb = workloads.bf16_bits(X)
        gn = g.cpu().numpy()
        ref = oracle.rmsnorm_mxcast(Xb, gn, 1e-6, B, FMTS[fmt])
        check_mx(Xb, gn, B, FMTS[fmt], (a.codes.cpu().numpy(), a.scales.cpu().numpy(), None),
                 ref, a.rinv.cpu().numpy(), 1e-6, f"fused {tag} {fmt} N={N} T={T}")


@pytest.mark.parametrize("fmt,B", [("e4m3", 32), ("nvfp4", 16)])
def test_fused_q_and_k_match_oracle(fmt, B):
    Q, gq = workloads.qk_inputs(333, 4096, seed=61, outlier_frac=0.01)
    K, gk = workloads.qk_inputs(333, 1024, seed=62)
    oq, ok = nts.qknorm_rms_qk_mxcast(Q.to(DEV), gq.to(DEV), K.to(DEV), gk.to(DEV), N=4, B=B,
                                      fmt=fmt, want_rinv=True)
    nts.check_status()
    for X, g, out, tag in ((Q, gq, oq, "Q"), (K, gk, ok, "K")):
        Xb = workloads.bf16_bits(X)
        gn = g.cpu().numpy()
        ref = oracle.rmsnorm_mxcast(Xb, gn, 1e-6, B, FMTS[fmt])
        check_mx(Xb, gn, B, FMTS[fmt], (out.codes.cpu().numpy(), out.scales.cpu().numpy(), None),
                 ref, out.rinv.cpu().numpy(), 1e-6, f"fused {tag} {fmt}")


def test_fused_q_and_k_arguments():
    Q, gq = workloads.qk_inputs(16, 1024, seed=63, device=DEV)
    K, gk = workloads.qk_inputs(16, 1000, seed=64, device=DEV)     # 1000/4 = 250: not a multiple of 32
    with pytest.raises(nts.NtsError, match="UNSUPPORTED"):
        nts.qknorm_rms_qk_mxcast(Q, gq, K, gk, N=4, B=32)
    K2, gk2 = workloads.qk_inputs(8, 1024, seed=65, device=DEV)
    with pytest.raises(ValueError):
        nts.qknorm_rms_qk_mxcast(Q, gq, K2, gk2, N=4, B=32)
    E = torch.empty(0, 1024, dtype=torch.bfloat16, device=DEV)
    oq, ok = nts.qknorm_rms_qk_mxcast(E, gq, E, gk2, N=2, B=32)
    nts.check_status()
    assert oq.codes.shape == (0, 1024) and ok.scales.shape == (0, 32)

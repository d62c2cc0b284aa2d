"""GPU parity of nts_layernorm_split (LayerNorm with two scalars per warp and
shard exchanged between cluster CTAs: the sum and M2 about the warp's own
mean, combined by the parallel-axis identity) against the oracle's
double-precision centred LayerNorm, through the C ABI.

Tolerances: the fp32 sums carry a relative error of a few 1e-7 per hundred
terms of the longest summation chain, so the mean is within about that times
mean|x|; M2 is formed about a mean close to the data, so the variance keeps
its relative accuracy whatever mu/sigma is (no cancellation of the one-pass
sum x^2/H - mu^2).  Per row:  |mu_g - mu_o| <= 1e-5 mean|x|,
|rstd_g/rstd_o - 1| <= 1e-5, and the bf16 outputs |g - o| <= 1e-3 + 1e-2 |o|
as for QK-RMSNorm.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import Y_ATOL, Y_RTOL, bf16_to_f64

pytestmark = pytest.mark.gpu

nts = pytest.importorskip("normalization_token_split_gb300")
DEV = "cuda:0"


def check_ln(X, Yg, mg, rg, Yo, mo, ro, what=""):
    x = bf16_to_f64(workloads.bf16_bits(X))
    mabs = np.abs(x).mean(axis=1)
    assert np.all(np.abs(mg - mo) <= 1e-5 * mabs + 1e-30), f"{what} mean"
    rel = np.abs(rg.astype(np.float64) / ro - 1.0)
    assert np.all(rel <= 1e-5), f"{what} rstd rel err {rel.max():.3g}"
    g, o = bf16_to_f64(Yg), bf16_to_f64(Yo)
    bad = np.abs(g - o) > Y_ATOL + Y_RTOL * np.abs(o)
    assert not bad.any(), f"{what} {bad.sum()} bf16 outputs out of tolerance"


def run_both(X, gamma, beta, eps, N, inplace=False):
    Xd = X.to(DEV)
    bd = None if beta is None else beta.to(DEV)
    Xb = workloads.bf16_bits(X)
    y, m, r = nts.layernorm_split(Xd, gamma.to(DEV), bd, eps=eps, N=N,
                                  out=Xd if inplace else None, want_stats=True)
    nts.check_status()
    Yo, mo, ro, _ = oracle.layernorm_split(Xb, gamma.cpu().numpy(),
                                           None if beta is None else beta.cpu().numpy(), eps, N)
    return workloads.bf16_bits(y), m.cpu().numpy(), r.cpu().numpy(), Yo, mo, ro


def test_tiny_split_config():
    X, g = workloads.qk_inputs(64, 1024, seed=400)
    b = workloads.beta_vector(1024, seed=400)
    Yg, mg, rg, Yo, mo, ro = run_both(X, g, b, 1e-5, 2)
    check_ln(X, Yg, mg, rg, Yo, mo, ro, "T=64 H=1024 N=2")


@pytest.mark.parametrize("H,N", [(64, 8), (128, 1), (1280, 2), (4096, 4), (5120, 8),
                                 (3072, 4), (24, 1), (8200, 1), (16384, 2), (30720, 1),
                                 (40960, 2)])
@pytest.mark.parametrize("T", [1, 3, 37, 513])
@pytest.mark.parametrize("with_beta", [True, False])
def test_shapes_and_ragged_tails(T, H, N, with_beta):
    X, g = workloads.qk_inputs(T, H, seed=T * 5 + H + N)
    b = workloads.beta_vector(H, seed=T + H) if with_beta else None
    if with_beta and H // N > 20480:
        # the shard's gamma and beta would not both fit in shared memory
        with pytest.raises(nts.NtsError, match="UNSUPPORTED"):
            nts.layernorm_split(X.to(DEV), g.to(DEV), b.to(DEV), N=N)
        return
    Yg, mg, rg, Yo, mo, ro = run_both(X, g, b, 1e-5, N)
    check_ln(X, Yg, mg, rg, Yo, mo, ro, f"T={T} H={H} N={N} beta={with_beta}")


@pytest.mark.parametrize("N", [1, 4, 8])
def test_prefill_full_size_with_outliers(N):
    X, g = workloads.qk_inputs(8192, 5120, seed=4100, outlier_frac=0.01, device=DEV)
    b = workloads.beta_vector(5120, seed=4100, device=DEV)
    Yg, mg, rg, Yo, mo, ro = run_both(X, g, b, 1e-5, N)
    check_ln(X, Yg, mg, rg, Yo, mo, ro, f"prefill N={N}")


def test_rows_with_a_large_mean():
    # mu = 3 sigma on most rows; rows 7 and 8 have mu/sigma ~ 10^3: values
    # 1000 (resp. -3008) plus or minus one bf16 step (4, resp. 16) with
    # probability 0.03 each way, sigma ~ 0.98 (3.9).  The one-pass variance
    # sum x^2/H - mu^2 would lose every digit to cancellation there.
    X, g = workloads.qk_inputs(256, 4096, seed=401)
    X = (X.float() + 3.0).to(torch.bfloat16)
    gen = torch.Generator().manual_seed(401)
    for r, (mu, step) in ((7, (1000.0, 4.0)), (8, (-3008.0, 16.0))):
        u = torch.rand(4096, generator=gen)
        b = torch.where(u < 0.03, -1.0, torch.where(u > 0.97, 1.0, 0.0))
        X[r] = (mu + step * b).to(torch.bfloat16)
        assert torch.equal(X[r].float(), mu + step * b)      # exact in bf16
    b = workloads.beta_vector(4096, seed=401)
    for N in (1, 4, 8):
        Yg, mg, rg, Yo, mo, ro = run_both(X, g, b, 1e-5, N)
        check_ln(X, Yg, mg, rg, Yo, mo, ro, f"large means N={N}")
        sigma = 1.0 / ro[7:9]
        assert np.all(np.abs(mo[7:9]) / sigma > 700)


def test_constant_and_zero_rows():
    # a constant row has zero variance: rstd = 1/sqrt(eps) and y = beta
    X, g = workloads.qk_inputs(16, 2048, seed=402)
    for r, c in enumerate((1.5, -0.75, 3.0, 0.0)):
        X[r] = c
    b = workloads.beta_vector(2048, seed=402)
    Yg, mg, rg, Yo, mo, ro = run_both(X, g, b, 1e-5, 4)
    check_ln(X, Yg, mg, rg, Yo, mo, ro, "constant rows")
    for r, c in enumerate((1.5, -0.75, 3.0, 0.0)):
        assert mg[r] == np.float32(c)
        # rstd = 1/sqrt(eps) up to the hardware rsqrt's rounding
        assert abs(rg[r] * np.sqrt(np.float64(np.float32(1e-5))) - 1) < 4e-7
        want = bf16_to_f64(workloads.bf16_bits(b.to(torch.bfloat16)))
        assert np.all(np.abs(bf16_to_f64(Yg[r]) - want) <= 1e-3 + 1e-2 * np.abs(want))


def test_in_place():
    X, g = workloads.qk_inputs(300, 4096, seed=403)
    b = workloads.beta_vector(4096, seed=403)
    Yg, mg, rg, Yo, mo, ro = run_both(X, g, b, 1e-5, 2, inplace=True)
    check_ln(X, Yg, mg, rg, Yo, mo, ro, "in place")


def test_no_beta_equals_zero_beta():
    X, g = workloads.qk_inputs(513, 4096, seed=404, device=DEV)
    z = torch.zeros(4096, device=DEV)
    y0, m0, r0 = nts.layernorm_split(X, g, None, N=4, want_stats=True)
    y1, m1, r1 = nts.layernorm_split(X, g, z, N=4, want_stats=True)
    nts.check_status()
    assert torch.equal(y0, y1) and torch.equal(m0, m1) and torch.equal(r0, r1)


def test_zero_tokens_and_no_stats():
    E = torch.empty(0, 1024, dtype=torch.bfloat16, device=DEV)
    g = torch.ones(1024, device=DEV)
    y, m, r = nts.layernorm_split(E, g, None, N=2, want_stats=True)
    nts.check_status()
    assert y.shape == (0, 1024) and m.shape == (0,)
    X, g = workloads.qk_inputs(100, 2048, seed=405, device=DEV)
    ya, _, _ = nts.layernorm_split(X, g, None, N=2)
    yb, _, _ = nts.layernorm_split(X, g, None, N=2, want_stats=True)
    nts.check_status()
    assert torch.equal(ya, yb)


@pytest.mark.parametrize("vpt,rows,stages,grid", [(1, 1, 1, 1), (2, 3, 2, 5), (8, 2, 4, 0),
                                                  (4, 7, 3, 7)])
def test_forced_launch_shapes(vpt, rows, stages, grid):
    X, g = workloads.qk_inputs(777, 2048, seed=406)
    b = workloads.beta_vector(2048, seed=406)
    try:
        nts.set_tuning(vpt=vpt, rows=rows, stages=stages, grid=grid)
        for N in (1, 4):
            Yg, mg, rg, Yo, mo, ro = run_both(X, g, b, 1e-5, N)
            check_ln(X, Yg, mg, rg, Yo, mo, ro, f"forced {vpt},{rows},{stages},{grid} N={N}")
    finally:
        nts.set_tuning()


def test_statistics_independent_of_N():
    X, g = workloads.qk_inputs(1024, 4096, seed=407, device=DEV)
    b = workloads.beta_vector(4096, seed=407, device=DEV)
    ref = nts.layernorm_split(X, g, b, N=1, want_stats=True)
    again = nts.layernorm_split(X, g, b, N=1, want_stats=True)
    nts.check_status()
    assert all(torch.equal(a, c) for a, c in zip(ref, again))      # deterministic
    for N in (2, 4, 8):
        y, m, r = nts.layernorm_split(X, g, b, N=N, want_stats=True)
        nts.check_status()
        assert torch.max(torch.abs(r / ref[2] - 1)) < 4e-6
        assert torch.max(torch.abs(m - ref[1])) < 1e-6

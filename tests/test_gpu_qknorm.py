"""GPU parity of nts_qknorm_rms against the oracle, through the C ABI.

Covers the layerwise QK-Norm workloads: the tiny split (T=64, H=1024, N=2),
the decode shapes (H=4096, T in {1,8,64,256}, N in {1,2,4,8}), the 13B-like
prefill with 1% outlier channels (H=5120, T=8192, N=4) at full size, edge
cases (T=0, ragged tails, narrow shards, in-place, all-zero rows, large
values) and properties (determinism, independence of N).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden
from parity import bf16_to_f64, check_qk

pytestmark = pytest.mark.gpu

nts = pytest.importorskip("normalization_token_split_gb300")
DEV = "cuda:0"


def run_gpu(X, gamma, eps, N, inplace=False):
    X = X.to(DEV)
    g = gamma.to(DEV)
    out = X if inplace else None
    Y, rinv = nts.qknorm_rms(X, g, eps=eps, N=N, out=out, want_rinv=True)
    nts.check_status()
    return workloads.bf16_bits(Y), rinv.cpu().numpy()


def run_both(X, gamma, eps, N, **kw):
    Yg, rg = run_gpu(X, gamma, eps, N, **kw)
    Yo, ro, _ = oracle.qknorm_rms(workloads.bf16_bits(X), gamma.cpu().numpy(), eps, N)
    return Yg, rg, Yo, ro


def test_tiny_split_config():
    X, g = workloads.qk_inputs(64, 1024, seed=0)
    Yg, rg, Yo, ro = run_both(X, g, 1e-6, 2)
    check_qk(Yg, rg, Yo, ro, "T=64 H=1024 N=2")


@pytest.mark.parametrize("T", [1, 8, 64, 256])
@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_decode_shapes(T, N):
    for which, seed in (("Q", 1000 + T), ("K", 2000 + T)):
        X, g = workloads.qk_inputs(T, 4096, seed=seed)
        Yg, rg, Yo, ro = run_both(X, g, 1e-6, N)
        check_qk(Yg, rg, Yo, ro, f"{which} T={T} N={N}")


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_prefill_full_size_with_outliers(N):
    # 13B-like prefill: Q and K each [8192, 5120], 1% of channels x20.
    for seed in (3000, 3001):
        X, g = workloads.qk_inputs(8192, 5120, seed=seed, outlier_frac=0.01, device=DEV)
        Yg, rg, Yo, ro = run_both(X, g, 1e-6, N)
        check_qk(Yg, rg, Yo, ro, f"prefill N={N}")


@pytest.mark.parametrize("H,N", [(64, 8), (128, 1), (1280, 2), (2048, 4), (5120, 8),
                                 (3072, 4), (640, 1), (24, 1), (8200, 1), (16384, 2),
                                 (30720, 1), (61440, 2)])
@pytest.mark.parametrize("T", [1, 3, 37, 513])
def test_shapes_and_ragged_tails(T, H, N):
    X, g = workloads.qk_inputs(T, H, seed=T * 7 + H + N)
    Yg, rg, Yo, ro = run_both(X, g, 1e-5, N)
    check_qk(Yg, rg, Yo, ro, f"T={T} H={H} N={N}")


def test_in_place():
    X, g = workloads.qk_inputs(300, 4096, seed=9)
    Yg, rg, Yo, ro = run_both(X, g, 1e-6, 4, inplace=True)
    check_qk(Yg, rg, Yo, ro, "in place")


def test_zero_rows_and_large_values():
    X, g = workloads.qk_inputs(64, 2048, seed=10)
    X[5] = 0
    X[6] = 3.0e4
    X[7, ::3] = -2.0e-30
    Yg, rg, Yo, ro = run_both(X, g, 1e-6, 2)
    check_qk(Yg, rg, Yo, ro, "degenerate rows")
    assert np.all(Yg[5] == 0) or np.all(bf16_to_f64(Yg[5]) == 0)


def test_worked_example_unsplit():
    # The SwiftQK notes' example (Sec. 4b) has 4-element shards, below the
    # kernel's 8-element vector; run it unsplit (N=1) as a single row.
    gd = read_golden("swiftqk_worked_example.txt")
    X = torch.tensor([gd["x"]], dtype=torch.float32).to(torch.bfloat16)
    g = torch.tensor(gd["gamma"], dtype=torch.float32)
    Yg, rg = run_gpu(X, g, gd["eps"], 1)
    assert abs(rg[0] - gd["rinv"]) < 0.5e-4
    y = bf16_to_f64(Yg[0])
    half_ulp = np.exp2(np.floor(np.log2(np.abs(gd["y"]))) - 8)
    assert np.all(np.abs(y - np.array(gd["y"])) <= half_ulp + gd["y_atol"])


def test_zero_tokens_launches_nothing():
    X = torch.empty(0, 1024, dtype=torch.bfloat16, device=DEV)
    g = torch.ones(1024, device=DEV)
    Y, r = nts.qknorm_rms(X, g, N=2, want_rinv=True)
    nts.check_status()
    assert Y.shape == (0, 1024)


def test_deterministic_and_independent_of_N():
    X, g = workloads.qk_inputs(1024, 4096, seed=11, device=DEV)
    outs = [run_gpu(X, g, 1e-6, N) for N in (1, 1, 2, 4, 8)]
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    for Yn, rn in outs[2:]:
        assert np.max(np.abs(rn / outs[0][1] - 1)) < 2e-6
        check_qk(Yn, rn, outs[0][0], outs[0][1].astype(np.float64), "N vs N=1")


@pytest.mark.parametrize("vpt,rows,stages,grid", [(1, 1, 1, 1), (2, 3, 2, 5), (8, 2, 4, 0),
                                                  (4, 7, 3, 7), (0, 0, 1, 0)])
def test_forced_launch_shapes(vpt, rows, stages, grid):
    X, g = workloads.qk_inputs(777, 2048, seed=12)
    try:
        nts.set_tuning(vpt=vpt, rows=rows, stages=stages, grid=grid)
        for N in (1, 4):
            Yg, rg, Yo, ro = run_both(X, g, 1e-6, N)
            check_qk(Yg, rg, Yo, ro, f"forced {vpt},{rows},{stages},{grid} N={N}")
    finally:
        nts.set_tuning()


def test_bounded_wait_reports_timeout_and_context_survives():
    X, g = workloads.qk_inputs(64, 1024, seed=13)
    try:
        nts.set_wait_limit_ns(20_000_000)     # 20 ms
        nts.set_missing_tx(16)                # first stage can never complete
        Xd, gd = X.to(DEV), g.to(DEV)
        nts.qknorm_rms(Xd, gd, N=2)
        with pytest.raises(nts.NtsError, match="TIMEOUT"):
            nts.check_status()
    finally:
        nts.set_missing_tx(0)
        nts.set_wait_limit_ns(0)
    # the context is still usable and the status word was cleared
    Yg, rg, Yo, ro = run_both(X, g, 1e-6, 2)
    check_qk(Yg, rg, Yo, ro, "after timeout")


def test_host_buffer_form():
    X, g = workloads.qk_inputs(500, 5120, seed=14)
    Xh = X.pin_memory()
    Yh = torch.empty_like(Xh).pin_memory()
    rh = torch.empty(500, dtype=torch.float32).pin_memory()
    Xd = torch.empty_like(X, device=DEV)
    Yd = torch.empty_like(X, device=DEV)
    rd = torch.empty(500, dtype=torch.float32, device=DEV)
    nts.qknorm_rms_host(Xh, g.to(DEV), Yh, Xd, Yd, eps=1e-6, N=4, rinv_host=rh, rinv_dev=rd)
    nts.check_status()
    Yo, ro, _ = oracle.qknorm_rms(workloads.bf16_bits(X), g.numpy(), 1e-6, 4)
    check_qk(workloads.bf16_bits(Yh), rh.numpy(), Yo, ro, "host form")


# ------------------------------------------------- fused Q+K single launch

@pytest.mark.parametrize("Hq,Hk", [(4096, 4096), (5120, 1024), (2048, 2048), (1024, 5120)])
@pytest.mark.parametrize("N", [1, 2, 4, 8])
@pytest.mark.parametrize("T", [1, 8, 256, 1031])
def test_fused_qk_matches_oracle(Hq, Hk, N, T):
    Q, gq = workloads.qk_inputs(T, Hq, seed=T + Hq, device=DEV)
    K, gk = workloads.qk_inputs(T, Hk, seed=T + Hk + 1, device=DEV)
    yq, yk, rq, rk = nts.qknorm_rms_qk(Q, gq, K, gk, eps=1e-6, N=N, want_rinv=True)
    nts.check_status()
    for X, g, Y, r in ((Q, gq, yq, rq), (K, gk, yk, rk)):
        Yo, ro, _ = oracle.qknorm_rms(workloads.bf16_bits(X), g.cpu().numpy(), 1e-6, N)
        check_qk(workloads.bf16_bits(Y), r.cpu().numpy(), Yo, ro, f"fused T={T} {Hq},{Hk} N={N}")


def test_fused_qk_prefill_full_size_equals_separate_calls():
    Q, gq = workloads.qk_inputs(8192, 5120, seed=3000, outlier_frac=0.01, device=DEV)
    K, gk = workloads.qk_inputs(8192, 5120, seed=3001, outlier_frac=0.01, device=DEV)
    yq, yk, rq, rk = nts.qknorm_rms_qk(Q, gq, K, gk, eps=1e-6, N=4, want_rinv=True)
    sq, srq = nts.qknorm_rms(Q, gq, eps=1e-6, N=4, want_rinv=True)
    sk, srk = nts.qknorm_rms(K, gk, eps=1e-6, N=4, want_rinv=True)
    nts.check_status()
    # same kernel arithmetic, same summation order: bit-identical
    assert torch.equal(yq, sq) and torch.equal(yk, sk)
    assert torch.equal(rq, srq) and torch.equal(rk, srk)
    Yo, ro, _ = oracle.qknorm_rms(workloads.bf16_bits(K), gk.cpu().numpy(), 1e-6, 4)
    check_qk(workloads.bf16_bits(yk), rk.cpu().numpy(), Yo, ro, "fused prefill K")


def test_fused_qk_in_place_and_zero_tokens():
    Q, gq = workloads.qk_inputs(300, 2048, seed=21, device=DEV)
    K, gk = workloads.qk_inputs(300, 1024, seed=22, device=DEV)
    Qb, Kb = workloads.bf16_bits(Q), workloads.bf16_bits(K)
    nts.qknorm_rms_qk(Q, gq, K, gk, eps=1e-6, N=2, out_q=Q, out_k=K, want_rinv=True)
    nts.check_status()
    for Xb, g, Y in ((Qb, gq, Q), (Kb, gk, K)):
        Yo, ro, _ = oracle.qknorm_rms(Xb, g.cpu().numpy(), 1e-6, 2)
        got, want = bf16_to_f64(workloads.bf16_bits(Y)), bf16_to_f64(Yo)
        assert np.all(np.abs(got - want) <= 1e-3 + 1e-2 * np.abs(want))
    E = torch.empty(0, 2048, dtype=torch.bfloat16, device=DEV)
    nts.qknorm_rms_qk(E, gq, E, gq, N=2)
    nts.check_status()


# ------------------------------------------------------- headwise QK-Norm

@pytest.mark.parametrize("T,H,hd,N", [(1, 4096, 128, 1), (37, 4096, 128, 1), (256, 2048, 64, 1),
                                      (129, 5120, 128, 2), (64, 1024, 256, 4), (8, 3072, 96, 1)])
def test_headwise_matches_oracle(T, H, hd, N):
    X, _ = workloads.qk_inputs(T, H, seed=T + H + hd)
    g = workloads.gamma_vector(hd, seed=hd)
    y, r = nts.qknorm_rms_heads(X.to(DEV), g.to(DEV), hd, eps=1e-6, N=N, want_rinv=True)
    nts.check_status()
    Yo, ro = oracle.qknorm_rms_heads(workloads.bf16_bits(X), g.numpy(), 1e-6, hd)
    check_qk(workloads.bf16_bits(y), r.cpu().numpy().ravel(), Yo, ro.ravel(), f"heads {T},{H},{hd},{N}")


@pytest.mark.parametrize("T,H,hd", [(1, 64, 8), (33, 512, 16), (100, 1024, 32), (513, 4096, 64),
                                    (7, 2048, 256), (3, 32768, 128), (300, 24, 8)])
def test_headwise_whole_heads_path(T, H, hd):
    # N = 1 keeps every head inside one CTA (segmented warp reduction)
    X, _ = workloads.qk_inputs(T, H, seed=T + 3 * H + hd, outlier_frac=0.02)
    g = workloads.gamma_vector(hd, seed=hd + 1)
    y, r = nts.qknorm_rms_heads(X.to(DEV), g.to(DEV), hd, eps=1e-6, N=1, want_rinv=True)
    nts.check_status()
    Yo, ro = oracle.qknorm_rms_heads(workloads.bf16_bits(X), g.numpy(), 1e-6, hd)
    check_qk(workloads.bf16_bits(y), r.cpu().numpy().ravel(), Yo, ro.ravel(), f"heads {T},{H},{hd}")


def test_headwise_prefill_full_size_sampled():
    X, _ = workloads.qk_inputs(8192, 5120, seed=3100, outlier_frac=0.01, device=DEV)
    g = workloads.gamma_vector(128, seed=128, device=DEV)
    y, r = nts.qknorm_rms_heads(X, g, 128, eps=1e-6, N=1, want_rinv=True)
    y2, r2 = nts.qknorm_rms_heads(X, g, 128, eps=1e-6, N=2, want_rinv=True)   # split heads
    nts.check_status()
    rows = torch.from_numpy(np.random.default_rng(5).choice(8192, 256, replace=False)).to(DEV)
    Yo, ro = oracle.qknorm_rms_heads(workloads.bf16_bits(X[rows]), g.cpu().numpy(), 1e-6, 128)
    check_qk(workloads.bf16_bits(y[rows]), r[rows].cpu().numpy().ravel(), Yo, ro.ravel(), "heads")
    check_qk(workloads.bf16_bits(y2[rows]), r2[rows].cpu().numpy().ravel(), Yo, ro.ravel(), "split")


@pytest.mark.parametrize("vpt,rows,stages,grid", [(1, 1, 1, 1), (2, 3, 2, 5), (8, 2, 4, 0),
                                                  (4, 7, 3, 7)])
def test_headwise_forced_launch_shapes(vpt, rows, stages, grid):
    X, _ = workloads.qk_inputs(777, 2048, seed=17)
    g = workloads.gamma_vector(128, seed=7)
    try:
        nts.set_tuning(vpt=vpt, rows=rows, stages=stages, grid=grid)
        y, r = nts.qknorm_rms_heads(X.to(DEV), g.to(DEV), 128, eps=1e-6, N=1, want_rinv=True)
        nts.check_status()
    finally:
        nts.set_tuning()
    Yo, ro = oracle.qknorm_rms_heads(workloads.bf16_bits(X), g.numpy(), 1e-6, 128)
    check_qk(workloads.bf16_bits(y), r.cpu().numpy().ravel(), Yo, ro.ravel(), "forced heads")


def test_headwise_bounded_wait_reports_timeout():
    X, _ = workloads.qk_inputs(64, 1024, seed=18)
    g = workloads.gamma_vector(128, seed=8)
    try:
        nts.set_wait_limit_ns(20_000_000)
        nts.set_missing_tx(16)
        nts.qknorm_rms_heads(X.to(DEV), g.to(DEV), 128, N=1)
        with pytest.raises(nts.NtsError, match="TIMEOUT"):
            nts.check_status()
    finally:
        nts.set_missing_tx(0)
        nts.set_wait_limit_ns(0)
    y, r = nts.qknorm_rms_heads(X.to(DEV), g.to(DEV), 128, eps=1e-6, N=1, want_rinv=True)
    nts.check_status()
    Yo, ro = oracle.qknorm_rms_heads(workloads.bf16_bits(X), g.numpy(), 1e-6, 128)
    check_qk(workloads.bf16_bits(y), r.cpu().numpy().ravel(), Yo, ro.ravel(), "after timeout")


# ------------------------------------------------- FP8-E4M3 activations

@pytest.mark.parametrize("T,H,N", [(1, 4096, 1), (64, 1024, 2), (257, 4096, 4), (33, 5120, 8),
                                   (8192, 5120, 4), (5, 16, 1), (100, 30720, 1)])
def test_fp8_input_matches_oracle(T, H, N):
    dev = DEV if T * H > 1 << 22 else "cpu"
    codes, scale, g = workloads.qk_inputs_fp8(T, H, seed=T + H, outlier_frac=0.01, device=dev)
    y, r = nts.qknorm_rms_fp8(codes.to(DEV), scale, g.to(DEV), eps=1e-6, N=N, want_rinv=True)
    nts.check_status()
    Yo, ro, _ = oracle.qknorm_rms_fp8(codes.cpu().numpy(), scale, g.cpu().numpy(), 1e-6, N)
    check_qk(workloads.bf16_bits(y), r.cpu().numpy(), Yo, ro, f"fp8 T={T} H={H} N={N}")


def test_fp8_equals_bf16_kernel_on_the_same_values():
    # E4M3 values are bf16 values: the FP8 kernel must match the bf16 kernel
    codes, scale, g = workloads.qk_inputs_fp8(512, 4096, seed=61, device=DEV)
    vals = (codes.view(torch.float8_e4m3fn).float() * scale).to(torch.bfloat16)
    y8, r8 = nts.qknorm_rms_fp8(codes, scale, g, eps=1e-6, N=4, want_rinv=True)
    yb, rb = nts.qknorm_rms(vals, g, eps=1e-6, N=4, want_rinv=True)
    nts.check_status()
    assert torch.equal(r8, rb) and torch.equal(y8, yb)


def test_headwise_tile_orders_agree():
    X, _ = workloads.qk_inputs(3001, 4096, seed=19, device=DEV)
    g = workloads.gamma_vector(128, seed=9, device=DEV)
    outs = []
    try:
        for dyn in (True, False, True):
            nts.set_schedule(dyn)
            for _ in range(3):
                y, r = nts.qknorm_rms_heads(X, g, 128, N=1, want_rinv=True)
            nts.check_status()
            outs.append((y, r))
    finally:
        nts.set_schedule(True)
    for y, r in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(r, outs[0][1])


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_cluster_tile_orders_agree(N):
    # dynamic order (rank 0 of each cluster takes tiles from the counter and
    # sends their numbers to its peers) and round-robin order: same results;
    # several back-to-back launches check that the counter re-arms itself
    Q, gq = workloads.qk_inputs(3001, 4096, seed=20 + N, device=DEV)
    K, gk = workloads.qk_inputs(3001, 1024, seed=30 + N, device=DEV)
    outs = []
    try:
        for dyn in (True, False, True):
            nts.set_schedule(dyn)
            for _ in range(3):
                res = nts.qknorm_rms_qk(Q, gq, K, gk, eps=1e-6, N=N, want_rinv=True)
                ln = nts.layernorm_split(Q, gq, None, N=N, want_stats=True)
            nts.check_status()
            outs.append(res + ln)
    finally:
        nts.set_schedule(True)
    for o in outs[1:]:
        assert all(torch.equal(a, b) for a, b in zip(o, outs[0]))
    Yo, ro, _ = oracle.qknorm_rms(workloads.bf16_bits(K), gk.cpu().numpy(), 1e-6, N)
    check_qk(workloads.bf16_bits(outs[0][1]), outs[0][3].cpu().numpy(), Yo, ro, f"dyn N={N}")


@pytest.mark.parametrize("T,H,N", [(8191, 5120, 4), (20000, 2048, 2)])
def test_host_buffer_form_in_chunks(T, H, N):
    X, g = workloads.qk_inputs(T, H, seed=T + H, outlier_frac=0.01)
    Xh = X.pin_memory()
    Yh = torch.empty_like(Xh).pin_memory()
    rh = torch.empty(T, dtype=torch.float32).pin_memory()
    Xd, Yd = torch.empty_like(X, device=DEV), torch.empty_like(X, device=DEV)
    rd = torch.empty(T, dtype=torch.float32, device=DEV)
    gd = g.to(DEV)
    for rep in range(2):
        nts.qknorm_rms_host(Xh, gd, Yh, Xd, Yd, eps=1e-6, N=N, rinv_host=rh, rinv_dev=rd)
        nts.check_status()
        y, r = nts.qknorm_rms(X.to(DEV), gd, eps=1e-6, N=N, want_rinv=True)
        nts.check_status()
        assert torch.equal(Yh, y.cpu()) and torch.equal(rh, r.cpu())
        Yh.zero_()


@pytest.mark.parametrize("T,Hq,Hk,N", [(8192, 5120, 5120, 4), (5000, 4096, 1024, 2), (7, 2048, 2048, 8)])
def test_fused_qk_host_buffer_form(T, Hq, Hk, N):
    # the host-buffer form of the fused Q+K launch (in chunks for the large
    # cases) equals the device form bit for bit, and the device form is
    # checked against the oracle elsewhere; two calls in a row
    Q, gq = workloads.qk_inputs(T, Hq, seed=T + Hq, outlier_frac=0.01)
    K, gk = workloads.qk_inputs(T, Hk, seed=T + Hk + 1, outlier_frac=0.01)
    Qh, Kh = Q.pin_memory(), K.pin_memory()
    Yqh, Ykh = torch.empty_like(Qh).pin_memory(), torch.empty_like(Kh).pin_memory()
    stage = [torch.empty_like(t, device=DEV) for t in (Q, Q, K, K)]
    gqd, gkd = gq.to(DEV), gk.to(DEV)
    yq, yk, _, rk = nts.qknorm_rms_qk(Q.to(DEV), gqd, K.to(DEV), gkd, eps=1e-6, N=N,
                                      want_rinv=True)
    nts.check_status()
    for rep in range(2):
        nts.qknorm_rms_qk_host(Qh, gqd, Yqh, Kh, gkd, Ykh, *stage, eps=1e-6, N=N)
        nts.check_status()
        assert torch.equal(Yqh, yq.cpu()) and torch.equal(Ykh, yk.cpu())
        Yqh.zero_()
        Ykh.zero_()
    Yo, ro, _ = oracle.qknorm_rms(workloads.bf16_bits(K[:64]), gk.numpy(), 1e-6, N)
    check_qk(workloads.bf16_bits(Ykh[:64].copy_(yk[:64].cpu())), rk[:64].cpu().numpy(), Yo, ro,
             "fused host form")


@pytest.mark.parametrize("N", [1, 2, 4, 8])
@pytest.mark.parametrize("T", [1, 3, 64, 200])
def test_decode_direct_kernel_equals_persistent(T, N):
    # decode-sized launches take the single-tile kernel; it must give the
    # persistent kernel's results bit for bit (same summation order)
    Q, gq = workloads.qk_inputs(T, 4096, seed=40 + T, device=DEV)
    K, gk = workloads.qk_inputs(T, 1024, seed=50 + T, device=DEV)
    outs = []
    try:
        for direct in (True, False):
            nts.set_direct(direct)
            r1 = nts.qknorm_rms_qk(Q, gq, K, gk, eps=1e-6, N=N, want_rinv=True)
            r2 = nts.qknorm_rms(Q, gq, eps=1e-6, N=N, want_rinv=True)
            nts.check_status()
            outs.append(r1 + r2)
    finally:
        nts.set_direct(True)
    assert all(torch.equal(a, b) for a, b in zip(outs[0], outs[1]))
    Yo, ro, _ = oracle.qknorm_rms(workloads.bf16_bits(Q), gq.cpu().numpy(), 1e-6, N)
    check_qk(workloads.bf16_bits(outs[0][4]), outs[0][5].cpu().numpy(), Yo, ro, f"direct N={N}")


@pytest.mark.parametrize("N", [1, 4])
@pytest.mark.parametrize("T", [1, 64])
def test_decode_direct_kernel_fp8_and_layernorm(T, N):
    codes, scale, g8 = workloads.qk_inputs_fp8(T, 4096, seed=60 + T, device=DEV)
    X, g = workloads.qk_inputs(T, 4096, seed=70 + T, device=DEV)
    b = workloads.beta_vector(4096, seed=70 + T, device=DEV)
    outs = []
    try:
        for direct in (True, False):
            nts.set_direct(direct)
            r8 = nts.qknorm_rms_fp8(codes, scale, g8, eps=1e-6, N=N, want_rinv=True)
            ln = nts.layernorm_split(X, g, b, N=N, want_stats=True)
            nts.check_status()
            outs.append(r8 + ln)
    finally:
        nts.set_direct(True)
    assert all(torch.equal(a, c) for a, c in zip(outs[0], outs[1]))
    Yo, ro, _ = oracle.qknorm_rms_fp8(codes.cpu().numpy(), scale, g8.cpu().numpy(), 1e-6, N)
    check_qk(workloads.bf16_bits(outs[0][0]), outs[0][1].cpu().numpy(), Yo, ro, f"fp8 direct N={N}")

"""Pins of the QK-RMSNorm oracle against what the pages and mathematics fix.

* The worked example of the SwiftQK reading notes, Sec. 4b, Eqs. (2)-(8)
  (tests/golden/swiftqk_worked_example.txt): exact shard sums, the global sum,
  RMS^-1 and the normalized shards.
* Closed form for a constant row x = c*1: y_j = gamma_j c / sqrt(c^2 + eps).
* Split-H equivalence (SwiftQK Sec. III.A; notes Sec. 4b, "identical up to
  the FP32 accumulation order"): shard sums add up to the unsplit sum and the
  output does not depend on N.
* Invariants of Eq. (1): scale invariance at eps = 0, equivariance under a
  joint permutation of columns and gains.
* The accuracy report of SwiftQK Sec. IV.C (bf16 vs an FP64 gold) as a
  sanity ceiling for the bf16 output.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden


def _bf16(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)


def _decode(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy().astype(np.float64)


def test_worked_example_eqs_2_to_8():
    g = read_golden("swiftqk_worked_example.txt")
    H, N = int(g["H"]), int(g["N"])
    X = workloads.bf16_bits(_bf16(g["x"]).reshape(1, H))
    Y, rinv, part = oracle.qknorm_rms(X, np.array(g["gamma"], np.float32), g["eps"], N)
    assert part[0, 0] == g["S0"] and part[0, 1] == g["S1"]          # Eqs. (3), (4)
    assert part[0].sum() == g["S"]                                   # Eq. (5)
    assert abs(rinv[0] - g["rinv"]) < 0.5 * 10 ** -g["rinv_digits"]  # Eq. (6)
    y = _decode(Y[0])
    half_ulp = np.exp2(np.floor(np.log2(np.abs(g["y"]))) - 8)
    assert np.all(np.abs(y - np.array(g["y"])) <= half_ulp + g["y_atol"])  # Eqs. (7), (8)


@pytest.mark.parametrize("N", [1, 2, 4])
def test_constant_row_closed_form(N):
    H = 64
    cs = [1.0, -3.0, 0.0078125, 0.5, 2.0 ** -10, 96.0]   # exact in bf16
    eps = 1e-6
    X = workloads.bf16_bits(workloads.constant_rows(len(cs), H, cs))
    gamma = workloads.gamma_vector(H, seed=11).numpy()
    Y, rinv, _ = oracle.qknorm_rms(X, gamma, eps, N)
    for t, c in enumerate(cs):
        r = 1.0 / np.sqrt(c * c + eps)
        assert rinv[t] == pytest.approx(r, rel=1e-15)
        want = gamma.astype(np.float64) * c * r
        got = _decode(Y[t])
        assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-300)


@pytest.mark.parametrize("N", [2, 4, 8])
def test_split_equals_unsplit(N):
    X, gamma = workloads.qk_inputs(16, 512, seed=5)
    Xb = workloads.bf16_bits(X)
    Y1, r1, p1 = oracle.qknorm_rms(Xb, gamma.numpy(), 1e-6, 1)
    YN, rN, pN = oracle.qknorm_rms(Xb, gamma.numpy(), 1e-6, N)
    assert np.allclose(pN.sum(axis=1), p1[:, 0], rtol=1e-12, atol=0)
    assert np.allclose(rN, r1, rtol=1e-12, atol=0)
    # the shards cover the row: each S_k is the sum over its own columns
    xd = _decode(Xb.ravel()).reshape(Xb.shape)
    W = 512 // N
    for k in range(N):
        assert np.allclose(pN[:, k], (xd[:, k * W:(k + 1) * W] ** 2).sum(axis=1), rtol=1e-12)
    # integer-valued rows: every partial sum is exact, so results are identical
    Xi = workloads.bf16_bits(torch.randint(-8, 9, (8, 512), generator=torch.Generator().manual_seed(3)).float().to(torch.bfloat16))
    Ya, ra, pa = oracle.qknorm_rms(Xi, gamma.numpy(), 1e-6, 1)
    Yb, rb, pb = oracle.qknorm_rms(Xi, gamma.numpy(), 1e-6, N)
    assert np.array_equal(ra, rb) and np.array_equal(Ya, Yb)
    assert np.array_equal(pb.sum(axis=1), pa[:, 0])


def test_scale_invariance_and_permutation():
    X, gamma = workloads.qk_inputs(8, 256, seed=6)
    Xb = workloads.bf16_bits(X)
    g = gamma.numpy()
    Y, _, _ = oracle.qknorm_rms(Xb, g, 0.0, 2)
    # x -> 4x is exact in bf16 and leaves Eq. (1) unchanged when eps = 0
    X4 = workloads.bf16_bits(X.float().mul(4.0).to(torch.bfloat16))
    Y4, _, _ = oracle.qknorm_rms(X4, g, 0.0, 2)
    assert np.array_equal(Y, Y4)
    # permuting columns of x and gamma together permutes y
    perm = np.random.default_rng(0).permutation(256)
    Yp, _, _ = oracle.qknorm_rms(np.ascontiguousarray(Xb[:, perm]), np.ascontiguousarray(g[perm]), 0.0, 1)
    assert np.array_equal(Yp, Y[:, perm])


def test_error_vs_fp64_gold_within_pages_bf16_report():
    # SwiftQK Sec. IV.C: bf16 activations, max abs error 5.0e-2 vs FP64 gold
    X, gamma = workloads.qk_inputs(64, 1024, seed=0)
    Xb = workloads.bf16_bits(X)
    Y, rinv, _ = oracle.qknorm_rms(Xb, gamma.numpy(), 1e-6, 2)
    xd = _decode(Xb.ravel()).reshape(Xb.shape)
    gold = xd * gamma.numpy().astype(np.float64) * rinv[:, None]
    err = np.abs(_decode(Y.ravel()).reshape(Y.shape) - gold)
    assert err.max() < 5.0e-2 and err.mean() < 2.1e-3 * 2


def test_degenerate_rows():
    # all-zero row: S = 0, RMS^-1 = 1/sqrt(eps), y = 0 (sign of x*gamma kept)
    X = workloads.bf16_bits(torch.zeros(2, 16, dtype=torch.bfloat16))
    Y, rinv, part = oracle.qknorm_rms(X, np.ones(16, np.float32), 1e-6, 4)
    assert np.all(part == 0) and np.allclose(rinv, 1e3, rtol=1e-12)
    assert np.all(Y == 0)
    # T = 0 is a no-op
    Y0, r0, p0 = oracle.qknorm_rms(np.zeros((0, 16), np.uint16), np.ones(16, np.float32), 1e-6, 2)
    assert Y0.shape == (0, 16) and r0.shape == (0,)


# ------------------------------------------------------- headwise QK-Norm

def test_headwise_single_head_is_layerwise():
    # with one head the headwise factor is the layerwise one (Sec. II.A)
    X, g = workloads.qk_inputs(16, 256, seed=31)
    Xb = workloads.bf16_bits(X)
    Yh, rh = oracle.qknorm_rms_heads(Xb, g.numpy(), 1e-6, 256)
    Yl, rl, _ = oracle.qknorm_rms(Xb, g.numpy(), 1e-6, 1)
    assert np.array_equal(Yh, Yl) and np.array_equal(rh[:, 0], rl)


def test_headwise_heads_are_independent_and_closed_form():
    T, hd, nh = 4, 32, 5
    g = workloads.gamma_vector(hd, seed=2).numpy()
    cs = np.array([[1.0, -2.0, 0.5, 4.0, 0.0], [3.0, 3.0, -0.25, 1.0, 8.0],
                   [0.125, 2.0, 2.0, -1.0, 1.0], [6.0, -6.0, 1.5, 0.75, -3.0]])
    x = np.repeat(cs, hd, axis=1)                      # every head constant
    Xb = workloads.bf16_bits(torch.tensor(x, dtype=torch.float32).to(torch.bfloat16))
    Y, r = oracle.qknorm_rms_heads(Xb, g, 1e-6, hd)
    assert np.allclose(r, 1 / np.sqrt(cs ** 2 + 1e-6), rtol=1e-14)
    want = (np.tile(g.astype(np.float64), nh) * x * np.repeat(r, hd, axis=1))
    got = _decode(Y.ravel()).reshape(Y.shape)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-300)
    # changing one head leaves the others bit-identical
    x2 = x.copy(); x2[:, 2 * hd:3 * hd] *= 3
    X2 = workloads.bf16_bits(torch.tensor(x2, dtype=torch.float32).to(torch.bfloat16))
    Y2, r2 = oracle.qknorm_rms_heads(X2, g, 1e-6, hd)
    keep = np.ones(nh * hd, bool); keep[2 * hd:3 * hd] = False
    assert np.array_equal(Y2[:, keep], Y[:, keep])
    assert np.array_equal(np.delete(r2, 2, axis=1), np.delete(r, 2, axis=1))


# ------------------------------------------------- FP8-E4M3 activations

def test_fp8_input_equals_bf16_path_on_the_same_values():
    # every E4M3 value is exactly a bf16 value: the FP8 oracle must equal the
    # (pinned) bf16 oracle fed the decoded values
    codes, scale, g = workloads.qk_inputs_fp8(32, 1024, seed=51)
    vals = codes.view(torch.float8_e4m3fn).float() * scale
    Xb = workloads.bf16_bits(vals.to(torch.bfloat16))
    assert np.array_equal(_decode(Xb.ravel()), vals.numpy().astype(np.float64).ravel())
    for N in (1, 2, 4):
        Y8, r8, p8 = oracle.qknorm_rms_fp8(codes.numpy(), scale, g.numpy(), 1e-6, N)
        Yb, rb, pb = oracle.qknorm_rms(Xb, g.numpy(), 1e-6, N)
        assert np.array_equal(Y8, Yb) and np.array_equal(r8, rb) and np.array_equal(p8, pb)


def test_fp8_scale_invariance_and_pages_error_report():
    codes, scale, g = workloads.qk_inputs_fp8(64, 1024, seed=52)
    Y1, _, _ = oracle.qknorm_rms_fp8(codes.numpy(), scale, g.numpy(), 0.0, 2)
    Y2, _, _ = oracle.qknorm_rms_fp8(codes.numpy(), scale * 8.0, g.numpy(), 0.0, 2)
    assert np.array_equal(Y1, Y2)
    # SwiftQK Sec. IV.C: FP8-E4M3 activations, max abs error 5.0e-1 vs FP64
    # gold; here the gold is Eq. (1) on the bf16 activations the FP8 codes
    # approximate
    X, gamma = workloads.qk_inputs(64, 1024, seed=52)
    Yo, _, _ = oracle.qknorm_rms(workloads.bf16_bits(X), gamma.numpy(), 1e-6, 2)
    Y8, _, _ = oracle.qknorm_rms_fp8(codes.numpy(), scale, g.numpy(), 1e-6, 2)
    err = np.abs(_decode(Y8.ravel()) - _decode(Yo.ravel()))
    assert err.max() < 5.0e-1 and err.mean() < 2.5e-2 * 2

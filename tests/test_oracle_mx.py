"""Pins of the MX-path oracle (RMSNorm + MXCast, MXNorm) against what the
MXNorm card and mathematics fix.

* Gaussian invariance (Fig. 1 caption: c(B, p) makes rho~ ~= rho for i.i.d.
  Gaussian rows), and the spread of rho~/rho shrinking like 1/sqrt(K) as the
  block count grows (Fig. 2 right: r^2 approaches 1 with more blocks).
* Closed forms on constant rows (all block absmaxes equal |c|).
* The block stage (Fig. 1 caption, Fig. A.1) re-derived by brute force: the
  scale exponent by search over all 255 E8M0 values of |log2 v - emax - e|,
  the element code by search over the format's whole value set (E4M3 values
  from torch's own float8 decoding; E2M1 from the OCP value table), ties to
  the even code, the E2M1 nibble layout, and the block absmax by numpy.
* The SwiftQK worked example through the RMSNorm + MXCast statistic.
* Invariants: scale invariance at eps = 0, gamma = None equals gamma = 1,
  power-mean inequality M_1 <= M_2.
* Where the gain enters each statistic (Fig. 1 caption: the left graph,
  RMSNorm + MXCast, takes its statistic from x as Eq. (1) of the SwiftQK
  notes does and applies the gain afterwards; the right graph, MXNorm, takes
  it from the block absmaxes of the tensor being cast, w = x*gamma):
  closed forms on constant rows with a constant gain g != 1, RMSNorm +
  MXCast's factor unchanged by any gain, and power-of-two gains that make
  w exactly representable in bf16, so that a call with the gain must equal
  a call without it on the pre-multiplied tensor.

MXCast semantics beyond these are unpinned by the pages (no worked MX example
is printed); the pins above are the definition's own consequences and the
library routines' encodings.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden

EMAX = {oracle.FMT_E4M3: 8, oracle.FMT_E2M1: 2}
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _decode_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).float().numpy()


def _format_table(fmt):
    """(positive magnitudes ascending, their codes) of the element format."""
    if fmt == oracle.FMT_E4M3:
        codes = np.arange(0, 0x7F, dtype=np.uint8)        # 0x7F is NaN
        vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    else:
        codes = np.arange(8, dtype=np.uint8)
        vals = E2M1_MAGNITUDES
    return vals, codes


def _nearest_codes(q, fmt):
    """Brute force: code of the nearest format value, ties to even code."""
    vals, codes = _format_table(fmt)
    a = np.minimum(np.abs(q), vals[-1])                    # saturating cast
    d = np.abs(a[:, None] - vals[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = (d == dmin)
    # prefer even codes among ties
    even = (codes & 1) == 0
    pick = np.where(cand & even[None, :], 1, 0) * 2 + cand
    idx = pick.argmax(axis=1)
    sign = np.signbit(q).astype(np.uint8) * (0x80 if fmt == oracle.FMT_E4M3 else 0x8)
    return codes[idx] | sign


def brute_force_block_stage(X, gamma, rinv, B, fmt):
    """Expected (codes, scales, amax) from the definition, searched exhaustively."""
    T, D = X.shape
    K = D // B
    x = _decode_bf16(X).astype(np.float32)
    w = x * gamma.astype(np.float32) if gamma is not None else x   # fp32 products
    wb = w.reshape(T, K, B).astype(np.float64)
    amax = np.abs(wb).max(axis=2)
    v = amax * rinv[:, None]
    cand = np.arange(-127, 128)
    with np.errstate(divide="ignore"):
        lv = np.log2(v)
    e = cand[np.argmin(np.abs(lv[..., None] - EMAX[fmt] - cand), axis=-1)]
    e = np.where(v > 0, e, -127)
    q = wb * rinv[:, None, None] * np.exp2(-e[..., None].astype(np.float64))
    codes = _nearest_codes(q.ravel(), fmt).reshape(T, D)
    if fmt == oracle.FMT_E2M1:
        codes = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return codes, (e + 127).astype(np.uint8), amax.astype(np.float32)


@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E2M1])
@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("kind", ["rms", "mx1", "mx2"])
def test_block_stage_brute_force(kind, B, fmt):
    X, gamma = workloads.mx_inputs(24, 256, seed=B + fmt, t_frac=0.2, with_gamma=True)
    Xb = workloads.bf16_bits(X)
    g = gamma.numpy()
    # a zero block and a tiny block exercise the clamped scale
    Xb[0, :B] = 0
    Xb[1, :B] = workloads.bf16_bits(torch.full((1, B), 1e-30).to(torch.bfloat16))
    if kind == "rms":
        codes, scales, rinv, amax = oracle.rmsnorm_mxcast(Xb, g, 1e-6, B, fmt)
    else:
        codes, scales, rinv, amax = oracle.mxnorm_cast(Xb, g, 1e-6, B, fmt, int(kind[-1]))
    c2, s2, a2 = brute_force_block_stage(Xb, g, rinv, B, fmt)
    assert np.array_equal(amax, a2)
    assert np.array_equal(scales, s2)
    assert np.array_equal(codes, c2)


def _rho_tilde_and_rho(D, B, p, T, seed):
    X, _ = workloads.mx_inputs(T, D, seed=seed)
    Xb = workloads.bf16_bits(X)
    _, _, rinv, _ = oracle.mxnorm_cast(Xb, None, 0.0, B, oracle.FMT_E4M3, p)
    x = _decode_bf16(Xb).astype(np.float64)
    rho = np.sqrt((x * x).mean(axis=1))
    return (1.0 / rinv) / rho


@pytest.mark.parametrize("D", [1024, 4096, 16384])
@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("p", [1, 2])
def test_gaussian_invariance(D, B, p):
    T = 8192 * 1024 // D
    ratio = _rho_tilde_and_rho(D, B, p, T, seed=D + B + p)
    assert abs(ratio.mean() - 1.0) <= 2e-3


def test_spread_shrinks_like_inverse_sqrt_blocks():
    s_small = _rho_tilde_and_rho(1024, 32, 2, 4096, seed=1).std()
    s_large = _rho_tilde_and_rho(16384, 32, 2, 512, seed=2).std()
    assert 3.0 < s_small / s_large < 5.3          # sqrt(16) = 4


@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E2M1])
def test_constant_rows_closed_form(B, p, fmt):
    cs = [1.0, -2.5, 0.0625, 40.0]
    D, eps = 4 * B, 1e-6
    Xb = workloads.bf16_bits(workloads.constant_rows(len(cs), D, cs))
    cB = oracle.mx_correction(B, p)
    _, scales, rinv, amax = oracle.mxnorm_cast(Xb, None, eps, B, fmt, p)
    _, scales_r, rinv_r, _ = oracle.rmsnorm_mxcast(Xb, None, eps, B, fmt)
    for t, c in enumerate(cs):
        assert np.all(amax[t] == abs(c))
        assert rinv[t] == pytest.approx(1 / math.sqrt((cB * c) ** 2 + eps), rel=1e-14)
        assert rinv_r[t] == pytest.approx(1 / math.sqrt(c * c + eps), rel=1e-14)
        # every block has absmax |c| r: one scale for the whole row
        assert len(set(scales[t])) == 1 and len(set(scales_r[t])) == 1


def test_worked_example_through_rmsnorm_statistic():
    g = read_golden("swiftqk_worked_example.txt")
    Xb = workloads.bf16_bits(torch.tensor(g["x"]).reshape(1, 8).to(torch.bfloat16))
    _, _, rinv, amax = oracle.rmsnorm_mxcast(Xb, None, g["eps"], 8, oracle.FMT_E4M3)
    assert abs(rinv[0] - g["rinv"]) < 0.5 * 10 ** -g["rinv_digits"]
    assert amax[0, 0] == 3.0


@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E2M1])
def test_invariants(fmt):
    X, _ = workloads.mx_inputs(16, 512, seed=9)
    Xb = workloads.bf16_bits(X)
    X4 = workloads.bf16_bits(X.float().mul(4.0).to(torch.bfloat16))
    for p in (1, 2):
        a = oracle.mxnorm_cast(Xb, None, 0.0, 32, fmt, p)
        b = oracle.mxnorm_cast(X4, None, 0.0, 32, fmt, p)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        c = oracle.mxnorm_cast(Xb, np.ones(512, np.float32), 0.0, 32, fmt, p)
        assert all(np.array_equal(u, v) for u, v in zip(a, c))
    r = oracle.rmsnorm_mxcast(Xb, None, 0.0, 32, fmt)
    r4 = oracle.rmsnorm_mxcast(X4, None, 0.0, 32, fmt)
    assert np.array_equal(r[0], r4[0]) and np.array_equal(r[1], r4[1])
    # power-mean inequality: M_1 <= M_2, i.e. (1/rinv)/c is larger for p = 2
    _, _, r1, _ = oracle.mxnorm_cast(Xb, None, 0.0, 32, fmt, 1)
    _, _, r2, _ = oracle.mxnorm_cast(Xb, None, 0.0, 32, fmt, 2)
    m1 = 1 / r1 / oracle.mx_correction(32, 1)
    m2 = 1 / r2 / oracle.mx_correction(32, 2)
    assert np.all(m1 <= m2 * (1 + 1e-15))


@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E2M1])
def test_given_rinv_stage_brute_force_and_agreement(fmt):
    X, gamma = workloads.mx_inputs(64, 1024, seed=21, t_frac=0.05, with_gamma=True)
    Xb, g = workloads.bf16_bits(X), gamma.numpy()
    codes, scales, rinv, amax = oracle.mxnorm_cast(Xb, g, 1e-6, 32, fmt, 2)
    r32 = rinv.astype(np.float32)
    c2, s2, a2 = oracle.mx_cast_given_rinv(Xb, g, r32, 32, fmt)
    assert np.array_equal(a2, amax)
    # brute force with the fp32 factor: scale decided on fl32(amax * r),
    # element values fl32(w * r)
    x = _decode_bf16(Xb).astype(np.float32)
    w = (x * g).reshape(64, 32, 32)
    v = (a2 * r32[:, None]).astype(np.float32).astype(np.float64)
    cand = np.arange(-127, 128)
    e = cand[np.argmin(np.abs(np.log2(v)[..., None] - EMAX[fmt] - cand), axis=-1)]
    assert np.array_equal(s2, (e + 127).astype(np.uint8))
    y = (w * r32[:, None, None]).astype(np.float32).astype(np.float64)
    q = y * np.exp2(-e[..., None].astype(np.float64))
    want = _nearest_codes(q.ravel(), fmt).reshape(64, 1024)
    if fmt == oracle.FMT_E2M1:
        want = (want[:, 0::2] | (want[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(c2, want)
    # the double-precision definition and the fp32 stage agree except at a
    # handful of rounding boundaries
    assert (scales != s2).mean() < 1e-3 and (codes != c2).mean() < 1e-3


def test_degenerate_rows():
    Xb = np.zeros((2, 64), np.uint16)
    for fmt in (oracle.FMT_E4M3, oracle.FMT_E2M1):
        codes, scales, rinv, amax = oracle.mxnorm_cast(Xb, None, 1e-6, 32, fmt, 2)
        assert np.all(codes == 0) and np.all(scales == 0) and np.allclose(rinv, 1e3)
        codes, scales, rinv, amax = oracle.rmsnorm_mxcast(Xb, None, 1e-6, 32, fmt)
        assert np.all(codes == 0) and np.all(scales == 0) and np.all(amax == 0)
    out = oracle.mxnorm_cast(np.zeros((0, 64), np.uint16), None, 1e-6, 32, 0, 2)
    assert out[0].shape == (0, 64)


# ----------------------------------------------------- post-round MXNorm

@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E2M1])
def test_postround_equals_preround_on_power_of_two_absmaxes(p, fmt):
    # blocks whose absmax is already a power of two are unchanged by rounding
    T, D, B = 12, 256, 32
    g = torch.Generator().manual_seed(41)
    powers = 2.0 ** torch.randint(-4, 5, (T, D // B), generator=g).float()
    u = (torch.rand(T, D // B, B, generator=g) * 1.8 - 0.9) * powers[..., None]
    u[..., 0] = powers * torch.where(torch.rand(T, D // B, generator=g) < 0.5, -1.0, 1.0)
    Xb = workloads.bf16_bits(u.reshape(T, D).to(torch.bfloat16))
    a = oracle.mxnorm_cast(Xb, None, 1e-6, B, fmt, p)
    b = oracle.mxnorm_postround_cast(Xb, None, 1e-6, B, fmt, p)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("p", [1, 2])
def test_postround_constant_rows_closed_form(p):
    # |c| = 3 rounds to 4 (3 > 2 sqrt 2); 1.25 to 1; 0.75 to 1 (> sqrt(2)/2);
    # 0.6875 to 0.5 (< sqrt(2)/2); 6 to 8
    cs = [3.0, -1.25, 0.75, 0.6875, 6.0]
    rounded = [4.0, 1.0, 1.0, 0.5, 8.0]
    Xb = workloads.bf16_bits(workloads.constant_rows(len(cs), 128, cs))
    cB = oracle.mx_correction(32, p)
    _, _, rinv, amax = oracle.mxnorm_postround_cast(Xb, None, 1e-6, 32, oracle.FMT_E4M3, p)
    for t, (c, a_hat) in enumerate(zip(cs, rounded)):
        assert np.all(amax[t] == abs(c))
        assert rinv[t] == pytest.approx(1 / math.sqrt((cB * a_hat) ** 2 + 1e-6), rel=1e-14)


def test_postround_estimate_within_sqrt2_of_preround():
    X, _ = workloads.mx_inputs(256, 1024, seed=42, t_frac=0.2)
    Xb = workloads.bf16_bits(X)
    for p in (1, 2):
        _, _, r_pre, _ = oracle.mxnorm_cast(Xb, None, 0.0, 32, oracle.FMT_E4M3, p)
        _, _, r_post, _ = oracle.mxnorm_postround_cast(Xb, None, 0.0, 32, oracle.FMT_E4M3, p)
        ratio = r_pre / r_post                      # = rho_post / rho_pre
        assert np.all(ratio >= 2 ** -0.5 * (1 - 1e-12)) and np.all(ratio <= 2 ** 0.5 * (1 + 1e-12))
        assert not np.allclose(ratio, 1.0)          # the rounding does change the estimate


# ---- the gain in the two statistics (Fig. 1 caption, left and right graphs)

@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E2M1])
@pytest.mark.parametrize("g", [3.0, 0.375, -2.0])
def test_constant_rows_with_constant_gain(B, p, fmt, g):
    # x = c*1 and gamma = g*1 with c*g exact in fp32: every block absmax of
    # w = x*gamma is |c*g|
    cs = [1.0, -2.5, 0.0625, 40.0]
    D, eps = 4 * B, 1e-6
    Xb = workloads.bf16_bits(workloads.constant_rows(len(cs), D, cs))
    gam = np.full(D, g, np.float32)
    cB = oracle.mx_correction(B, p)
    _, _, rinv_m, amax_m = oracle.mxnorm_cast(Xb, gam, eps, B, fmt, p)
    _, _, rinv_r, amax_r = oracle.rmsnorm_mxcast(Xb, gam, eps, B, fmt)
    for t, c in enumerate(cs):
        assert np.all(amax_m[t] == abs(c * g)) and np.all(amax_r[t] == abs(c * g))
        # MXNorm: the estimate comes from the absmaxes of w
        assert rinv_m[t] == pytest.approx(1 / math.sqrt((cB * c * g) ** 2 + eps), rel=1e-14)
        # RMSNorm + MXCast: the statistic is of x, whatever the gain
        assert rinv_r[t] == pytest.approx(1 / math.sqrt(c * c + eps), rel=1e-14)


@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E2M1])
def test_rmsnorm_factor_does_not_depend_on_the_gain(fmt):
    X, gam = workloads.mx_inputs(32, 1024, seed=41, t_frac=0.1, with_gamma=True)
    Xb = workloads.bf16_bits(X)
    _, _, r_g, amax_g = oracle.rmsnorm_mxcast(Xb, gam.numpy(), 1e-6, 32, fmt)
    _, _, r_0, amax_0 = oracle.rmsnorm_mxcast(Xb, None, 1e-6, 32, fmt)
    assert np.array_equal(r_g, r_0)                  # bit for bit
    assert not np.array_equal(amax_g, amax_0)        # while the cast tensor differs


def _pow2_gain_and_premultiplied(T, D, seed):
    """A gain of powers of two (per channel, both signs) and bf16(x*gamma),
    which equals fp32(x*gamma) exactly: scaling a bf16 value by 2^k stays in
    bf16 while the exponent stays in range."""
    X, _ = workloads.mx_inputs(T, D, seed=seed, t_frac=0.1)
    gen = torch.Generator().manual_seed(seed)
    k = torch.randint(-3, 4, (D,), generator=gen).float()
    sign = torch.where(torch.rand(D, generator=gen) < 0.3, -1.0, 1.0)
    gam = (sign * torch.pow(2.0, k)).float()
    W = (X.float() * gam).to(torch.bfloat16)
    assert torch.equal(W.float(), X.float() * gam)
    return workloads.bf16_bits(X), gam.numpy(), workloads.bf16_bits(W)


@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E2M1])
def test_mxnorm_statistic_is_of_the_cast_tensor(B, p, fmt):
    Xb, gam, Wb = _pow2_gain_and_premultiplied(24, 16 * B, seed=B + 10 * p + fmt)
    with_gain = oracle.mxnorm_cast(Xb, gam, 1e-6, B, fmt, p)
    premult = oracle.mxnorm_cast(Wb, None, 1e-6, B, fmt, p)
    for u, v in zip(with_gain, premult):
        assert np.array_equal(u, v)
    # and the gain does change the result (the pin is not vacuous)
    plain = oracle.mxnorm_cast(Xb, None, 1e-6, B, fmt, p)
    assert not np.array_equal(with_gain[2], plain[2])


@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E2M1])
@pytest.mark.parametrize("k", [-3, 2, 5])
def test_power_of_two_gain_shifts_only_the_rmsnorm_scales(B, fmt, k):
    # gamma = 2^k on every channel: w = 2^k x exactly.  RMSNorm + MXCast keeps
    # the factor of x, so w*rinv is 2^k times the ungained values: the element
    # codes stay, every E8M0 scale moves up by exactly k.  MXNorm (eps = 0)
    # estimates its factor from w, which cancels the gain: nothing changes.
    X, _ = workloads.mx_inputs(24, 16 * B, seed=B + k, t_frac=0.1)
    Xb = workloads.bf16_bits(X)
    gam = np.full(16 * B, 2.0 ** k, np.float32)
    c_g, s_g, r_g, a_g = oracle.rmsnorm_mxcast(Xb, gam, 1e-6, B, fmt)
    c_0, s_0, r_0, a_0 = oracle.rmsnorm_mxcast(Xb, None, 1e-6, B, fmt)
    assert np.array_equal(r_g, r_0)
    assert np.array_equal(a_g, a_0 * np.float32(2.0 ** k))
    assert np.array_equal(c_g, c_0)
    assert np.array_equal(s_g.astype(int), s_0.astype(int) + k)
    for p in (1, 2):
        m_g = oracle.mxnorm_cast(Xb, gam, 0.0, B, fmt, p)
        m_0 = oracle.mxnorm_cast(Xb, None, 0.0, B, fmt, p)
        assert np.array_equal(m_g[0], m_0[0]) and np.array_equal(m_g[1], m_0[1])
        assert np.allclose(m_g[2] * 2.0 ** k, m_0[2], rtol=1e-15, atol=0)

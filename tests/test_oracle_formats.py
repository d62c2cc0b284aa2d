"""Pins of the oracle's number formats and of c(B, p), against things other
than the oracle itself: torch's own casts (library routines), exhaustive
nearest-value search over the format's value set, double-precision log2, and
closed forms / scipy quadrature of the order-statistic moment.

Sources: OCP Microscaling Formats v1.0 (E4M3, E2M1, E8M0 encodings); MXNorm
card, Fig. 1 caption (absmax / 2^emax, power-of-two rounding 2^round(log2),
correction factor c(B, p) making the estimate exact for Gaussian inputs).
"""
import math

import numpy as np
import pytest
import torch

import oracle


# --------------------------------------------------------------------------
# bfloat16
# --------------------------------------------------------------------------

def test_bf16_matches_torch_cast():
    rng = np.random.default_rng(1)
    # random fp32 values over a wide exponent range, plus every midpoint
    # between neighbouring bf16 values and its fp32 neighbours
    f = (rng.standard_normal(200_000) * np.exp2(rng.integers(-60, 60, 200_000))).astype(np.float32)
    hi = np.arange(0, 0x7F80, dtype=np.uint32) << 16        # all finite positive bf16
    mid = ((hi + 0x8000)).view(np.float32)                  # exact midpoints
    mids = np.concatenate([mid, np.nextafter(mid, np.float32(np.inf)),
                           np.nextafter(mid, np.float32(0))])
    vals = np.concatenate([f, mids, -mids]).astype(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) < 3.3e38)]
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.to_bf16(vals.astype(np.float64))
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# E4M3
# --------------------------------------------------------------------------

def _e4m3_table():
    codes = np.arange(256, dtype=np.uint8)
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def test_e4m3_decoder_matches_torch():
    tab = _e4m3_table()
    for c in range(256):
        d = oracle.decode(c, oracle.FMT_E4M3)
        if math.isnan(tab[c]):
            assert math.isnan(d)
        else:
            assert d == tab[c] and math.copysign(1, d) == math.copysign(1, tab[c])


def test_e4m3_encoder_exhaustive_vs_torch():
    # every bf16 bit pattern in range, every E4M3 midpoint and its fp32
    # neighbours; torch's float32 -> float8_e4m3fn cast is round-to-nearest-even
    allbf = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    tab = _e4m3_table()
    pos = np.unique(tab[(tab >= 0) & np.isfinite(tab)])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0))])
    vals = np.concatenate([allbf, near, -near]).astype(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448.0)]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.encode(vals.astype(np.float64), oracle.FMT_E4M3)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_e4m3_saturates_and_keeps_sign_of_zero():
    got = oracle.encode([1000.0, -1000.0, 449.0, 470.0, -0.0, 0.0, -1e-30], oracle.FMT_E4M3)
    assert list(got) == [0x7E, 0xFE, 0x7E, 0x7E, 0x80, 0x00, 0x80]


# --------------------------------------------------------------------------
# E2M1
# --------------------------------------------------------------------------

E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # OCP table, codes 0..7


def test_e2m1_decoder_table():
    for c in range(16):
        mag = E2M1_MAGNITUDES[c & 7]
        d = oracle.decode(c, oracle.FMT_E2M1)
        assert abs(d) == mag and (math.copysign(1, d) < 0) == bool(c & 8)


def _nearest_even(v, values, codes_even):
    """Brute-force round-to-nearest, ties to the code with even LSB."""
    dist = np.abs(values - v)
    best = np.flatnonzero(dist == dist.min())
    if len(best) > 1:
        best = [b for b in best if codes_even[b]]
    return best[0]


def test_e2m1_encoder_brute_force():
    mags = np.array(E2M1_MAGNITUDES)
    even = np.array([(c & 1) == 0 for c in range(8)])
    rng = np.random.default_rng(2)
    mids = (mags[:-1] + mags[1:]) / 2
    vals = np.concatenate([mids, np.nextafter(mids, 10), np.nextafter(mids, 0),
                           rng.uniform(0, 7, 5000), [0.0, 6.0, 6.5, 100.0]])
    got = oracle.encode(vals, oracle.FMT_E2M1)
    for v, g in zip(vals, got):
        want = _nearest_even(min(v, 6.0), mags, even)     # satfinite clamps at 6
        assert g == want, (v, g, want)
    neg = oracle.encode(-vals, oracle.FMT_E2M1)
    assert np.array_equal(neg, got | 0x8)


def test_e2m1_ties_to_even_examples():
    got = oracle.encode([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], oracle.FMT_E2M1)
    assert [E2M1_MAGNITUDES[c] for c in got] == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


# --------------------------------------------------------------------------
# E8M0 (power-of-two rounding in the log2 domain)
# --------------------------------------------------------------------------

def test_round_log2_against_double_log2_on_every_fp32_exponent():
    # mantissas either side of sqrt(2) and at the ends of the binade
    mants = np.array([0x000000, 0x3504F3, 0x3504F4, 0x7FFFFF, 0x123456, 0x6A09E6], np.uint32)
    exps = np.arange(1, 255, dtype=np.uint32)
    bits = (exps[:, None] << 23 | mants[None, :]).ravel()
    v = bits.view(np.float32).astype(np.float64)
    # an fp32 m is at least 2.5e-8 away from sqrt(2); double log2 resolves it
    want = np.rint(np.log2(v)).astype(np.int64)
    got = np.array([oracle.round_log2(x) for x in v])
    assert np.array_equal(got, want)
    m = bits & 0x7FFFFF
    e = (bits >> 23).astype(np.int64) - 127
    assert np.array_equal(got, e + (m >= 0x3504F4))


def test_e8m0_exponent_brute_force_and_clamp():
    rng = np.random.default_rng(3)
    v = np.exp2(rng.uniform(-140, 140, 20000))
    for emax in (8, 2):
        got = oracle.e8m0_exponent(v, emax)
        cand = np.arange(-127, 128)
        want = np.array([cand[np.argmin(np.abs(np.log2(x) - emax - cand))] for x in v])
        assert np.array_equal(got, want)
    assert list(oracle.e8m0_exponent([0.0, 1e-300, 2.0 ** 200], 8)) == [-127, -127, 127]


# --------------------------------------------------------------------------
# c(B, p)
# --------------------------------------------------------------------------

def test_correction_closed_forms():
    # B = 1: E|Z| = sqrt(2/pi), E Z^2 = 1.
    assert oracle.mx_correction(1, 1) == pytest.approx(math.sqrt(math.pi / 2), rel=1e-10)
    assert oracle.mx_correction(1, 2) == pytest.approx(1.0, rel=1e-10)
    # B = 2: E max(|Z1|,|Z2|) = 2/sqrt(pi); E max(Z1^2, Z2^2) = 1 + 2/pi.
    assert oracle.mx_correction(2, 1) == pytest.approx(math.sqrt(math.pi) / 2, rel=1e-10)
    assert oracle.mx_correction(2, 2) == pytest.approx(1 / math.sqrt(1 + 2 / math.pi), rel=1e-10)


@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("p", [1, 2])
def test_correction_vs_scipy_density_form(B, p):
    from scipy import integrate, special
    # E[M^p] = int x^p * d/dx erf(x/sqrt2)^B dx  (density form; the oracle
    # integrates the survival form)
    dens = lambda x: x ** p * B * special.erf(x / math.sqrt(2)) ** (B - 1) * math.sqrt(2 / math.pi) * math.exp(-x * x / 2)
    m, _ = integrate.quad(dens, 0, 40, limit=400, epsabs=1e-14, epsrel=1e-13)
    assert oracle.mx_correction(B, p) == pytest.approx(m ** (-1 / p), rel=1e-9)


def test_correction_monte_carlo():
    rng = np.random.default_rng(4)
    z = np.abs(rng.standard_normal((400_000, 32))).max(axis=1)
    for p in (1, 2):
        mc = np.mean(z ** p) ** (-1 / p)
        assert oracle.mx_correction(32, p) == pytest.approx(mc, rel=3e-3)

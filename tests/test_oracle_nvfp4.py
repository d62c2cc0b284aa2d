"""Pins of the oracle's NVFP4 block stage (E2M1 values, 16-value blocks, one
E4M3 scale per block; the MXNorm card lists NVFP4 among its kernel cases,
Table 4, and the stage's rules are this build's reading): a closed form for
constant rows, brute-force nearest-value searches for every scale and every
element code, saturation, zero blocks, and the format independence of the
MXNorm statistic."""
import numpy as np
import pytest
import torch

import oracle
import workloads

F4, E4, NV = oracle.FMT_E2M1, oracle.FMT_E4M3, oracle.FMT_NVFP4
E4M3_VALUES = np.array([oracle.decode(c, E4) for c in range(0x7F)])     # finite, >= 0
E2M1_VALUES = np.array([oracle.decode(c, F4) for c in range(8)])


def nearest_even(table, v):
    """Index of the nearest table entry to v >= 0 (ties to the even index),
    saturating at the last entry: a brute-force search."""
    d = np.abs(table - v)
    best = np.flatnonzero(d == d.min())
    return int(best[0] if len(best) == 1 or best[0] % 2 == 0 else best[1])


def unpack(codes, D):
    out = np.empty((codes.shape[0], D), np.uint8)
    out[:, 0::2] = codes & 0xF
    out[:, 1::2] = codes >> 4
    return out


def test_constant_rows_closed_form():
    # RMSNorm of a constant row c gives y = c / sqrt(c^2 + eps) ~ sign(c); the
    # block scale is the E4M3 value nearest 1/6, 0.171875 (code 0x23), and
    # y / s = 5.82 rounds to the E2M1 value 6 (code 7, sign bit 8).
    X = torch.tensor([[1.0] * 64, [-3.0] * 64], dtype=torch.bfloat16)
    codes, scales, r, amax = oracle.rmsnorm_mxcast(workloads.bf16_bits(X), None, 1e-6, 16, NV)
    assert oracle.decode(0x23, E4) == 0.171875
    assert np.all(scales == 0x23)
    q = unpack(codes, 64)
    assert np.all(q[0] == 0x7) and np.all(q[1] == 0xF)


@pytest.mark.parametrize("fn", ["rms", "mx1", "mx2"])
def test_scales_and_codes_are_brute_force_nearest_values(fn):
    X, _ = workloads.mx_inputs(12, 256, seed=81, t_frac=0.5)
    Xb = workloads.bf16_bits(X)
    if fn == "rms":
        codes, scales, r, amax = oracle.rmsnorm_mxcast(Xb, None, 1e-6, 16, NV)
    else:
        codes, scales, r, amax = oracle.mxnorm_cast(Xb, None, 1e-6, 16, NV, int(fn[-1]))
    x = X.double().numpy()
    q = unpack(codes, 256)
    for t in range(12):
        for k in range(16):
            blk = x[t, 16 * k:16 * k + 16]
            a = np.abs(blk).max()
            assert amax[t, k] == np.float32(a)
            sc = nearest_even(E4M3_VALUES, a * r[t] / 6.0)
            assert scales[t, k] == sc
            s = E4M3_VALUES[sc]
            for b in range(16):
                y = blk[b] * r[t]
                mag = nearest_even(E2M1_VALUES, abs(y) / s)
                want = mag | (8 if np.signbit(y) else 0)
                assert q[t, 16 * k + b] == want, (t, k, b)


def test_saturation_and_zero_blocks():
    X = torch.zeros(2, 32, dtype=torch.bfloat16)
    X[0, :16] = torch.linspace(-1, 1, 16)
    X[1, 16:] = -0.0                      # a zero block of negative zeros
    Xb = workloads.bf16_bits(X)
    # a huge factor drives amax*r/6 past 448: the scale saturates to 448
    codes, scales, amax = oracle.mx_cast_given_rinv(Xb, None, np.array([1e6, 1.0], np.float32),
                                                    16, NV)
    assert scales[0, 0] == 0x7E and oracle.decode(0x7E, E4) == 448.0
    q = unpack(codes, 32)
    assert q[0, 0] == 0xF and q[0, 15] == 0x7          # -6 and +6, saturated
    # zero blocks: scale code 0 and +0 codes, whatever the sign of the zeros
    assert scales[0, 1] == 0 and np.all(q[0, 16:] == 0)
    assert np.all(scales[1] == 0) and np.all(q[1] == 0)


def test_statistic_does_not_depend_on_the_element_format():
    X, _ = workloads.mx_inputs(20, 512, seed=82, t_frac=0.3)
    Xb = workloads.bf16_bits(X)
    for p in (1, 2):
        _, _, r_nv, a_nv = oracle.mxnorm_cast(Xb, None, 1e-6, 16, NV, p)
        _, _, r_f4, a_f4 = oracle.mxnorm_cast(Xb, None, 1e-6, 16, F4, p)
        assert np.array_equal(r_nv, r_f4) and np.array_equal(a_nv, a_f4)
    _, _, r_nv, _ = oracle.rmsnorm_mxcast(Xb, None, 1e-6, 16, NV)
    _, _, r_e4, _ = oracle.rmsnorm_mxcast(Xb, None, 1e-6, 16, E4)
    assert np.array_equal(r_nv, r_e4)


def test_fp32_stage_matches_double_definition_away_from_midpoints():
    X, g = workloads.mx_inputs(64, 1024, seed=83, with_gamma=True)
    Xb = workloads.bf16_bits(X)
    c_d, s_d, r, _ = oracle.rmsnorm_mxcast(Xb, g.numpy(), 1e-6, 16, NV)
    c_f, s_f, _ = oracle.mx_cast_given_rinv(Xb, g.numpy(), r.astype(np.float32), 16, NV)
    assert np.mean(s_d == s_f) > 0.999 and np.mean(c_d == c_f) > 0.999


def test_rejects_other_block_sizes_and_post_round():
    X = workloads.bf16_bits(torch.ones(1, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        oracle.rmsnorm_mxcast(X, None, 1e-6, 32, NV)
    with pytest.raises(ValueError):
        oracle.mxnorm_postround_cast(X, None, 1e-6, 16, NV, 2)

"""Property tests of the oracle over random small shapes (T, H, N, B, format,
statistic and the seed of the values drawn from a seeded generator, one
draw per test case, so the same cases run wherever the suite runs).

Properties that follow from the definitions alone:

* QK-RMSNorm (SwiftQK Eq. (1)): negating the row negates every output bit
  for bit and leaves rinv unchanged; the split into N shards changes the
  double-precision statistic only by rounding (the two-stage sum equals the
  unsplit one, SwiftQK Sec. III.A); permuting a row's columns together with
  gamma permutes the outputs.
* RMSNorm + MXCast and MXNorm (MXNorm card, Fig. 1 caption): negating the
  row flips the sign bit of every element code and changes neither the
  scales, the absmaxes nor rinv; the block absmax is the largest |x * gamma|
  of the block in fp32; reordering whole blocks reorders scales and codes
  (MXNorm's statistic is a sum over blocks, so rinv moves only by rounding).
"""
import numpy as np
import pytest

import oracle


FMTS = [oracle.FMT_E4M3, oracle.FMT_E2M1]
SIGN = {oracle.FMT_E4M3: 0x80, oracle.FMT_E2M1: 0x88}


def bf16_rows(T, H, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H)).astype(np.float32) * np.float32(scale)
    return oracle.to_bf16(x).reshape(T, H)


def gamma_vec(H, seed):
    rng = np.random.default_rng(seed + 1)
    return (1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32)


def qk_shape(case):
    """(T, N, shard width / 8, seed) of a QK case."""
    rng = np.random.default_rng(1000 + case)
    return (int(rng.integers(1, 6)), int(rng.choice([1, 2, 4, 8])), int(rng.integers(1, 9)),
            int(rng.integers(0, 2**31 - 1)))


def mx_shape(case):
    """(T, B, blocks, format, statistic, with gamma, seed) of an MX case."""
    rng = np.random.default_rng(2000 + case)
    return (int(rng.integers(1, 5)), int(rng.choice([16, 32, 64])), int(rng.integers(1, 7)),
            FMTS[int(rng.integers(0, 2))], int(rng.integers(0, 3)), bool(rng.integers(0, 2)),
            int(rng.integers(0, 2**31 - 1)))


@pytest.mark.parametrize("case", range(60))
def test_qk_sign_symmetry(case):
    shape = qk_shape(case)
    T, N, w8, seed = shape
    H = N * 8 * w8
    X = bf16_rows(T, H, seed)
    g = gamma_vec(H, seed)
    Y, r, _ = oracle.qknorm_rms(X, g, 1e-6, N)
    Yn, rn, _ = oracle.qknorm_rms(X ^ np.uint16(0x8000), g, 1e-6, N)
    assert np.array_equal(Yn, Y ^ np.uint16(0x8000))
    assert np.array_equal(rn, r)


@pytest.mark.parametrize("case", range(60))
def test_qk_split_only_reorders_the_sum(case):
    shape = qk_shape(case)
    T, N, w8, seed = shape
    H = N * 8 * w8
    X = bf16_rows(T, H, seed)
    g = gamma_vec(H, seed)
    _, r1, p1 = oracle.qknorm_rms(X, g, 1e-6, 1)
    _, rN, pN = oracle.qknorm_rms(X, g, 1e-6, N)
    assert np.allclose(pN.sum(axis=1), p1[:, 0], rtol=1e-13, atol=0)
    assert np.allclose(rN, r1, rtol=1e-13, atol=0)


@pytest.mark.parametrize("case", range(40))
def test_qk_column_permutation(case):
    shape = qk_shape(case)
    T, N, w8, seed = shape
    H = N * 8 * w8
    X = bf16_rows(T, H, seed)
    g = gamma_vec(H, seed)
    perm = np.random.default_rng(seed + 2).permutation(H)
    Y, r, _ = oracle.qknorm_rms(X, g, 1e-6, N)
    Yp, rp, _ = oracle.qknorm_rms(np.ascontiguousarray(X[:, perm]), g[perm], 1e-6, N)
    assert np.allclose(rp, r, rtol=1e-13, atol=0)
    # one rounding to bf16 of values equal up to ~1e-16: at most one bf16 ulp
    diff = np.abs(Yp.astype(np.int32) - Y[:, perm].astype(np.int32))
    assert diff.max() <= 1


def run_mx(X, g, B, fmt, p):
    if p == 0:
        return oracle.rmsnorm_mxcast(X, g, 1e-6, B, fmt)
    return oracle.mxnorm_cast(X, g, 1e-6, B, fmt, p)


@pytest.mark.parametrize("case", range(60))
def test_mx_sign_symmetry(case):
    shape = mx_shape(case)
    T, B, K, fmt, p, with_gamma, seed = shape
    D = B * K
    X = bf16_rows(T, D, seed, scale=3.0)
    g = gamma_vec(D, seed) if with_gamma else None
    c, s, r, a = run_mx(X, g, B, fmt, p)
    cn, sn, rn, an = run_mx(X ^ np.uint16(0x8000), g, B, fmt, p)
    assert np.array_equal(sn, s) and np.array_equal(rn, r) and np.array_equal(an, a)
    assert np.array_equal(cn, c ^ np.uint8(SIGN[fmt]))


@pytest.mark.parametrize("case", range(60))
def test_mx_block_absmax_is_the_largest_weighted_magnitude(case):
    shape = mx_shape(case)
    T, B, K, fmt, p, with_gamma, seed = shape
    D = B * K
    X = bf16_rows(T, D, seed, scale=3.0)
    g = gamma_vec(D, seed) if with_gamma else None
    _, _, _, a = run_mx(X, g, B, fmt, p)
    x = (X.astype(np.uint32) << 16).view(np.float32)
    w = x if g is None else (x * g).astype(np.float32)
    want = np.abs(w).reshape(T, K, B).max(axis=2)
    assert np.array_equal(a, want)


@pytest.mark.parametrize("case", range(40))
def test_mx_block_permutation(case):
    shape = mx_shape(case)
    T, B, K, fmt, p, with_gamma, seed = shape
    D = B * K
    X = bf16_rows(T, D, seed, scale=3.0)
    g = gamma_vec(D, seed) if with_gamma else None
    bperm = np.random.default_rng(seed + 3).permutation(K)
    cols = (bperm[:, None] * B + np.arange(B)[None, :]).reshape(-1)
    c, s, r, a = run_mx(X, g, B, fmt, p)
    cp, sp, rp, ap = run_mx(np.ascontiguousarray(X[:, cols]), None if g is None else g[cols],
                            B, fmt, p)
    assert np.array_equal(ap, a[:, bperm])
    assert np.allclose(rp, r, rtol=1e-13, atol=0)
    # the codes and scales are decided with the (double) rinv: compare where
    # that rinv is the same to the last bit (reordering a sum rarely moves it)
    same = rp == r
    if fmt == oracle.FMT_E4M3:
        cperm = c.reshape(T, K, B)[:, bperm].reshape(T, D)
    else:
        cperm = c.reshape(T, K, B // 2)[:, bperm].reshape(T, D // 2)
    assert np.array_equal(sp[same], s[same][:, bperm])
    assert np.array_equal(cp[same], cperm[same])

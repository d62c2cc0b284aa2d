"""Pins of the split-H LayerNorm oracle (SwiftQK reading notes, Sec. 5e:
LayerNorm's statistics are two additive scalars per shard, sum x and
sum x^2, combined like RMSNorm's single sum of squares)."""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _decode(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).float().numpy().astype(np.float64)


def test_constant_row_gives_beta():
    # x = c*1: mu = c, var = 0, y = beta exactly (closed form)
    H = 64
    g = workloads.gamma_vector(H, 1).numpy()
    b = workloads.gamma_vector(H, 2).numpy() - 1.0
    Xb = workloads.bf16_bits(workloads.constant_rows(3, H, [2.0, -5.0, 0.0]))
    Y, mu, r, _ = oracle.layernorm_split(Xb, g, b, 1e-5, 4)
    assert np.allclose(mu, [2.0, -5.0, 0.0], rtol=0, atol=0)
    assert np.allclose(r, 1 / np.sqrt(1e-5), rtol=1e-12)
    assert np.array_equal(Y, np.tile(oracle.to_bf16(b.astype(np.float64)), (3, 1)))


@pytest.mark.parametrize("N", [2, 4, 8])
def test_shard_sums_add_up_and_split_equals_unsplit(N):
    X, g = workloads.qk_inputs(16, 512, seed=71)
    Xb = workloads.bf16_bits(X)
    b = np.linspace(-1, 1, 512).astype(np.float32)
    Y1, m1, r1, p1 = oracle.layernorm_split(Xb, g.numpy(), b, 1e-5, 1)
    YN, mN, rN, pN = oracle.layernorm_split(Xb, g.numpy(), b, 1e-5, N)
    x = _decode(Xb.ravel()).reshape(16, 512)
    W = 512 // N
    for k in range(N):
        assert np.allclose(pN[:, k, 0], x[:, k * W:(k + 1) * W].sum(1), rtol=1e-12, atol=1e-12)
        assert np.allclose(pN[:, k, 1], (x[:, k * W:(k + 1) * W] ** 2).sum(1), rtol=1e-12)
    assert np.allclose(pN.sum(1), p1[:, 0], rtol=1e-12, atol=1e-12)
    assert np.allclose(mN, m1, rtol=1e-12, atol=1e-15) and np.allclose(rN, r1, rtol=1e-12)
    assert np.array_equal(YN, Y1)


def test_two_scalar_identity_and_invariances():
    # var computed from the two additive scalars equals the centred definition
    X, g = workloads.qk_inputs(32, 1024, seed=72)
    Xb = workloads.bf16_bits(X)
    _, mu, r, part = oracle.layernorm_split(Xb, g.numpy(), None, 0.0, 4)
    S1, S2 = part.sum(1)[:, 0], part.sum(1)[:, 1]
    var2 = S2 / 1024 - (S1 / 1024) ** 2
    assert np.allclose(1 / r ** 2, var2, rtol=1e-10)
    # shift by a constant (exact in bf16 for these values) leaves y unchanged
    Xi = torch.randint(-16, 17, (8, 256), generator=torch.Generator().manual_seed(3)).float()
    A = workloads.bf16_bits(Xi.to(torch.bfloat16))
    Bb = workloads.bf16_bits((Xi + 64.0).to(torch.bfloat16))
    gg = workloads.gamma_vector(256, 3).numpy()
    Ya, *_ = oracle.layernorm_split(A, gg, None, 0.0, 2)
    Yb, *_ = oracle.layernorm_split(Bb, gg, None, 0.0, 2)
    assert np.array_equal(Ya, Yb)
    # scale by 4 leaves y unchanged at eps = 0
    C = workloads.bf16_bits((Xi * 4.0).to(torch.bfloat16))
    Yc, *_ = oracle.layernorm_split(C, gg, None, 0.0, 2)
    assert np.array_equal(Ya, Yc)
    # output rows have mean beta-free 0 and unit variance (gamma = 1)
    Y1, *_ = oracle.layernorm_split(A, np.ones(256, np.float32), None, 0.0, 1)
    y = _decode(Y1.ravel()).reshape(8, 256)
    assert np.allclose(y.mean(1), 0, atol=2e-3) and np.allclose(y.std(1), 1, atol=5e-3)

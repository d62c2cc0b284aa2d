"""Seeded synthetic inputs for the per-token normalization paths.

This module holds no arithmetic of the method itself: it only draws random
activations and gains with torch's seeded generators and rounds them to
bfloat16.  Both the CPU oracle (via the tests and the benchmark) and the CUDA
path consume its outputs; neither side imports the other.

Recipes (the pages' workloads, restated as synthetic inputs):

* QK-Norm (SwiftQK micro-benchmarks: Q/K widths 1024-5120, 64 and 4096
  tokens; 13B-like prefill with outlier channels):
  X ~ N(0, 1) rounded to bf16, optionally with a seeded fraction of channels
  (columns) multiplied by 20 before rounding; gamma ~ N(1, 0.1) in fp32.
* MX paths (MXNorm card, Table 4 kernel grid):
  X ~ N(0, 1) rounded to bf16, optionally with a seeded Bernoulli fraction of
  rows replaced by Student-t(3) draws (heavy-tailed rows); gamma, when used,
  ~ N(1, 0.1).  A Student-t(df) draw is Z0 / sqrt(chi2_df / df) with chi2_df
  the sum of df squared standard normals.

Values drawn on a CUDA device differ from those drawn on the CPU for the same
seed (different generators); every consumer takes the tensors as produced and
copies them where needed, so each check compares like with like.
"""
from __future__ import annotations

import numpy as np
import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """bfloat16 tensor (any device) -> numpy uint16 bit patterns on the host."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def gamma_vector(n: int, seed: int, device="cpu") -> torch.Tensor:
    """gamma ~ N(1, 0.1) in fp32."""
    g = _gen(seed * 7919 + 17, device)
    return 1.0 + 0.1 * torch.randn(n, generator=g, device=device, dtype=torch.float32)


def qk_inputs(T: int, H: int, seed: int, outlier_frac: float = 0.0,
              outlier_scale: float = 20.0, device="cpu"):
    """(X bf16 [T,H], gamma fp32 [H]) for the QK-Norm path."""
    g = _gen(seed, device)
    x = torch.randn(T, H, generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0.0 and H > 0:
        gc = _gen(seed * 31 + 5, "cpu")
        n_out = max(1, int(round(outlier_frac * H)))
        cols = torch.randperm(H, generator=gc)[:n_out].to(device)
        x[:, cols] *= outlier_scale
    return x.to(torch.bfloat16), gamma_vector(H, seed, device)


def beta_vector(H: int, seed: int, device="cpu") -> torch.Tensor:
    """LayerNorm shift beta fp32 [H]: small values around zero."""
    g = _gen(seed * 7 + 3, device)
    return 0.1 * torch.randn(H, generator=g, device=device, dtype=torch.float32)


def outlier_columns(H: int, seed: int, outlier_frac: float) -> np.ndarray:
    """The columns qk_inputs scales for the given seed (for reporting)."""
    gc = _gen(seed * 31 + 5, "cpu")
    n_out = max(1, int(round(outlier_frac * H)))
    return torch.randperm(H, generator=gc)[:n_out].numpy()


def mx_inputs(T: int, D: int, seed: int, t_frac: float = 0.0, df: int = 3,
              with_gamma: bool = False, device="cpu"):
    """(X bf16 [T,D], gamma fp32 [D] or None) for the MX paths."""
    g = _gen(seed, device)
    x = torch.randn(T, D, generator=g, device=device, dtype=torch.float32)
    if t_frac > 0.0 and T > 0:
        gc = _gen(seed * 131 + 7, "cpu")
        rows = torch.nonzero(torch.rand(T, generator=gc) < t_frac).flatten().to(device)
        if rows.numel():
            z = torch.randn(rows.numel(), D, generator=g, device=device)
            chi2 = torch.zeros_like(z)
            for _ in range(df):
                chi2 += torch.randn(rows.numel(), D, generator=g, device=device) ** 2
            x[rows] = z / torch.sqrt(chi2 / df)
    gamma = gamma_vector(D, seed, device) if with_gamma else None
    return x.to(torch.bfloat16), gamma


def student_t_rows(T: int, seed: int, t_frac: float) -> np.ndarray:
    """Row indices mx_inputs draws from Student-t for the given seed."""
    gc = _gen(seed * 131 + 7, "cpu")
    return torch.nonzero(torch.rand(T, generator=gc) < t_frac).flatten().numpy()


def constant_rows(T: int, D: int, values, device="cpu") -> torch.Tensor:
    """Rows x = c * 1 (one constant per row), as bf16."""
    c = torch.as_tensor(values, dtype=torch.float32, device=device).reshape(T, 1)
    return (c * torch.ones(T, D, device=device)).to(torch.bfloat16)


def qk_inputs_fp8(T: int, H: int, seed: int, outlier_frac: float = 0.0, device="cpu"):
    """(X E4M3 codes uint8 [T,H], x_scale, gamma fp32 [H]) for the FP8-input
    QK-Norm: the bf16 recipe of qk_inputs divided by a per-tensor scale
    (absmax / 448, rounded to a power of two) and cast with torch's
    float8_e4m3fn conversion."""
    x, gamma = qk_inputs(T, H, seed, outlier_frac=outlier_frac, device=device)
    xf = x.float()
    amax = float(xf.abs().max()) if xf.numel() else 1.0
    scale = 2.0 ** np.ceil(np.log2(max(amax, 1e-30) / 448.0))
    codes = (xf / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, float(scale), gamma

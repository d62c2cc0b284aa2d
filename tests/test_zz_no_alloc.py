"""nts_mxnorm_cast_host_noalloc: the host-buffer MXNorm entry point whose
device staging is the library's fixed array.  Compared with the existing
entry points on two calls in a row (the second call reuses the array the
first one left behind).  Collected last on purpose: it must pass both in a
fresh process and after every other test."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

nts = pytest.importorskip("normalization_token_split_gb300")
DEV = "cuda:0"


def host_outputs(T, D, B, fmt):
    cb = D if fmt == "e4m3" else D // 2
    return (torch.empty(T, cb, dtype=torch.uint8).pin_memory(),
            torch.empty(T, D // B, dtype=torch.uint8).pin_memory())


@pytest.mark.parametrize("T,D,B,fmt,p,with_gamma", [
    (1024, 4096, 32, "e4m3", 2, False),
    (777, 2048, 16, "nvfp4", 1, True),
    (3, 1040, 16, "e2m1", 2, False),
    (513, 3072, 64, "e4m3", 1, True),
])
def test_matches_existing_entry_points_on_two_calls_in_a_row(T, D, B, fmt, p, with_gamma):
    for seed in (1, 2):      # two calls in a row through the shared array
        X, g = workloads.mx_inputs(T, D, seed=970 + seed + T, t_frac=0.05, with_gamma=with_gamma)
        Xh = X.pin_memory()
        gh = g.pin_memory() if with_gamma else None
        codes_h, scales_h = host_outputs(T, D, B, fmt)
        nts.mxnorm_cast_host_noalloc(Xh, gh, codes_h, scales_h, eps=1e-6, B=B, fmt=fmt, p=p)
        torch.cuda.synchronize()
        nts.check_status()
        ref = nts.mxnorm_cast(X.to(DEV), None if g is None else g.to(DEV), eps=1e-6, B=B,
                              fmt=fmt, p=p)
        ref_h = host_outputs(T, D, B, fmt)
        nts.mxnorm_cast_host(Xh, None if g is None else g.to(DEV), ref_h[0], ref_h[1],
                             X.to(DEV), torch.empty_like(ref.codes), torch.empty_like(ref.scales),
                             eps=1e-6, B=B, fmt=fmt, p=p)
        torch.cuda.synchronize()
        nts.check_status()
        assert torch.equal(codes_h, ref.codes.cpu()) and torch.equal(scales_h, ref.scales.cpu())
        assert torch.equal(codes_h, ref_h[0]) and torch.equal(scales_h, ref_h[1])


def test_refuses_calls_beyond_the_array():
    X = torch.zeros(4096, 4096, dtype=torch.bfloat16)     # 32 MiB of X alone
    codes_h, scales_h = host_outputs(4096, 4096, 32, "e4m3")
    with pytest.raises(nts.NtsError, match="static scratch"):
        nts.mxnorm_cast_host_noalloc(X, None, codes_h, scales_h, B=32)

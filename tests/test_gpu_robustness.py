"""Checks that stand in for a memory checker and a fault injector (neither
runs on this GPU pool), through the C ABI:

* canaries: every output is placed inside a larger buffer filled with a
  fixed byte; after the call the bytes before and after it must be
  unchanged, and the output must equal that of a call on a plain buffer
  (an out-of-bounds store of any kernel shows up as a changed canary);
* injected launch failures: the library's launch-failure hook makes a call
  fail the way a failed launch would, and the next calls run normally;
* random shapes: seeded random token counts, widths, shard counts, block
  sizes, formats and statistics, each against the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_mx, check_qk

pytestmark = pytest.mark.gpu

nts = pytest.importorskip("normalization_token_split_gb300")
DEV = "cuda:0"
PAD = 4096          # canary bytes on each side (keeps 16-byte alignment)
CANARY = 0xA5
FMTS = {"e4m3": oracle.FMT_E4M3, "e2m1": oracle.FMT_E2M1, "nvfp4": oracle.FMT_NVFP4}


class Padded:
    """A tensor of `shape` and `dtype` inside a canary-filled byte buffer."""

    def __init__(self, shape, dtype):
        self.n = math.prod(shape) * torch.tensor([], dtype=dtype).element_size()
        self.buf = torch.full((2 * PAD + self.n,), CANARY, dtype=torch.uint8, device=DEV)
        self.t = self.buf[PAD:PAD + self.n].view(dtype).view(shape)

    def intact(self):
        return bool((self.buf[:PAD] == CANARY).all()) and bool(
            (self.buf[PAD + self.n:] == CANARY).all())


def check_canaries(outs, what):
    nts.check_status()
    for name, p in outs.items():
        assert p.intact(), f"{what}: bytes around {name} changed"


@pytest.mark.parametrize("T,H,N", [(1, 1024, 2), (37, 5120, 4), (513, 4096, 8), (300, 24, 1),
                                   (1000, 2048, 2), (4097, 1280, 4)])
def test_canaries_split_h_paths(T, H, N):
    X, g = workloads.qk_inputs(T, H, seed=T + H + N, device=DEV)
    b = workloads.beta_vector(H, seed=1, device=DEV)
    Y, r = Padded((T, H), torch.bfloat16), Padded((T,), torch.float32)
    nts.qknorm_rms(X, g, N=N, out=Y.t, rinv=r.t)
    check_canaries({"Y": Y, "rinv": r}, f"qknorm_rms T={T} H={H} N={N}")
    ref, rr = nts.qknorm_rms(X, g, N=N, want_rinv=True)
    assert torch.equal(Y.t, ref) and torch.equal(r.t, rr)

    K, gk = workloads.qk_inputs(T, H // 2 if (H // 2) % (8 * N) == 0 else H, seed=5, device=DEV)
    Yq, Yk = Padded(tuple(X.shape), torch.bfloat16), Padded(tuple(K.shape), torch.bfloat16)
    rq, rk = Padded((T,), torch.float32), Padded((T,), torch.float32)
    nts.qknorm_rms_qk(X, g, K, gk, N=N, out_q=Yq.t, out_k=Yk.t, rinv_q=rq.t, rinv_k=rk.t)
    check_canaries({"Yq": Yq, "Yk": Yk, "rinv_q": rq, "rinv_k": rk}, "qknorm_rms_qk")

    Y2, m, s = (Padded((T, H), torch.bfloat16), Padded((T,), torch.float32),
                Padded((T,), torch.float32))
    nts.layernorm_split(X, g, b, N=N, out=Y2.t, mean=m.t, rstd=s.t)
    check_canaries({"Y": Y2, "mean": m, "rstd": s}, "layernorm_split")

    if (H // N) % 16 == 0:
        codes8, scale8, g8 = workloads.qk_inputs_fp8(T, H, seed=3, device=DEV)
        Y3 = Padded((T, H), torch.bfloat16)
        nts.qknorm_rms_fp8(codes8, scale8, g8, N=N, out=Y3.t)
        check_canaries({"Y": Y3}, "qknorm_rms_fp8")

    for fmt, B in (("e4m3", 32), ("nvfp4", 16), ("e2m1", 64)):
        if (H // N) % B:
            continue
        cb = H if fmt == "e4m3" else H // 2
        c, sc, r2 = (Padded((T, cb), torch.uint8), Padded((T, H // B), torch.uint8),
                     Padded((T,), torch.float32))
        nts.qknorm_rms_mxcast(X, g, N=N, B=B, fmt=fmt, codes=c.t, scales=sc.t, rinv=r2.t)
        check_canaries({"codes": c, "scales": sc, "rinv": r2}, f"qknorm_rms_mxcast {fmt}")
        ref = nts.qknorm_rms_mxcast(X, g, N=N, B=B, fmt=fmt)
        assert torch.equal(c.t, ref.codes) and torch.equal(sc.t, ref.scales)


@pytest.mark.parametrize("T,H,hd", [(1, 4096, 128), (77, 2048, 64), (1000, 5120, 128)])
def test_canaries_headwise(T, H, hd):
    X, _ = workloads.qk_inputs(T, H, seed=T + H, device=DEV)
    g = workloads.gamma_vector(hd, seed=3, device=DEV)
    Y, r = Padded((T, H), torch.bfloat16), Padded((T, H // hd), torch.float32)
    nts.qknorm_rms_heads(X, g, hd, out=Y.t, rinv=r.t)
    check_canaries({"Y": Y, "rinv": r}, f"heads T={T} H={H}")


@pytest.mark.parametrize("T,D,fmt,B", [
    (T, D, fmt, B)
    for T, D in [(1, 256), (37, 1024), (333, 4096), (2001, 1040), (5, 16384)]
    for fmt, B in [("e4m3", 32), ("e2m1", 16), ("nvfp4", 16), ("e4m3", 64), ("e2m1", 64)]
    if D % B == 0])
def test_canaries_mx_paths(T, D, fmt, B):
    X, g = workloads.mx_inputs(T, D, seed=T + D + B, with_gamma=True)
    X, g = X.to(DEV), g.to(DEV)
    cb = D if fmt == "e4m3" else D // 2
    calls = [("rms", lambda **o: nts.rmsnorm_mxcast(X, g, B=B, fmt=fmt, **o)),
             ("mx p=2", lambda **o: nts.mxnorm_cast(X, None, B=B, fmt=fmt, p=2, **o)),
             ("mx p=1", lambda **o: nts.mxnorm_cast(X, g, B=B, fmt=fmt, p=1, **o))]
    if fmt != "nvfp4":
        calls.append(("post", lambda **o: nts.mxnorm_postround_cast(X, None, B=B, fmt=fmt, p=2,
                                                                    **o)))
    for name, call in calls:
        c, s = Padded((T, cb), torch.uint8), Padded((T, D // B), torch.uint8)
        r, a = Padded((T,), torch.float32), Padded((T, D // B), torch.float32)
        call(codes=c.t, scales=s.t, rinv=r.t, amax=a.t)
        check_canaries({"codes": c, "scales": s, "rinv": r, "amax": a}, f"{name} {fmt} B={B}")
        ref = call(want_rinv=True, want_amax=True)
        nts.check_status()
        assert torch.equal(c.t, ref.codes) and torch.equal(s.t, ref.scales)
        assert torch.equal(r.t, ref.rinv) and torch.equal(a.t, ref.amax)


def test_injected_launch_failure_and_recovery():
    X, g = workloads.qk_inputs(300, 2048, seed=71, device=DEV)
    want, _ = nts.qknorm_rms(X, g, N=2)
    Xm, _ = workloads.mx_inputs(300, 2048, seed=72, device=DEV)
    want_mx = nts.mxnorm_cast(Xm, None, B=32, p=2)
    try:
        nts.inject_failure("CUDA", 2)
        with pytest.raises(nts.NtsError, match="NTS_ERR_CUDA.*injected"):
            nts.qknorm_rms(X, g, N=2)
        with pytest.raises(nts.NtsError, match="NTS_ERR_CUDA.*injected"):
            nts.mxnorm_cast(Xm, None, B=32, p=2)
        nts.inject_failure("TIMEOUT", 1)
        with pytest.raises(nts.NtsError, match="NTS_ERR_TIMEOUT"):
            nts.qknorm_rms_qk(X, g, X, g, N=2)
    finally:
        nts.inject_failure("CUDA", 0)
    nts.check_status()
    got, _ = nts.qknorm_rms(X, g, N=2)
    got_mx = nts.mxnorm_cast(Xm, None, B=32, p=2)
    nts.check_status()
    assert torch.equal(got, want)
    assert torch.equal(got_mx.codes, want_mx.codes) and torch.equal(got_mx.scales, want_mx.scales)


def test_injected_failure_inside_a_chunked_host_call():
    # the first chunk's kernel "fails": the call reports it, and the next
    # host-buffer call (same internal copy streams) runs normally
    T, D = 9000, 2048
    X, _ = workloads.mx_inputs(T, D, seed=73)
    Xh = X.pin_memory()
    ch = torch.empty(T, D, dtype=torch.uint8).pin_memory()
    sh = torch.empty(T, D // 32, dtype=torch.uint8).pin_memory()
    Xd = torch.empty_like(X, device=DEV)
    cd = torch.empty(T, D, dtype=torch.uint8, device=DEV)
    sd = torch.empty(T, D // 32, dtype=torch.uint8, device=DEV)
    try:
        nts.inject_failure("CUDA", 1)
        with pytest.raises(nts.NtsError, match="injected"):
            nts.mxnorm_cast_host(Xh, None, ch, sh, Xd, cd, sd, B=32, p=2)
    finally:
        nts.inject_failure("CUDA", 0)
    torch.cuda.synchronize()
    nts.mxnorm_cast_host(Xh, None, ch, sh, Xd, cd, sd, B=32, p=2)
    nts.check_status()
    ref = nts.mxnorm_cast(X.to(DEV), None, B=32, p=2)
    nts.check_status()
    assert torch.equal(ch, ref.codes.cpu()) and torch.equal(sh, ref.scales.cpu())


def test_random_shapes_split_h():
    rng = np.random.default_rng(20261202)
    for case in range(40):
        N = int(rng.choice([1, 2, 4, 8]))
        W = 8 * int(rng.integers(1, 200))
        T = int(rng.integers(1, 700))
        eps = float(rng.choice([1e-6, 1e-5, 1e-3]))
        X, g = workloads.qk_inputs(T, N * W, seed=1000 + case, outlier_frac=0.01)
        Y, r = nts.qknorm_rms(X.to(DEV), g.to(DEV), eps=eps, N=N, want_rinv=True)
        nts.check_status()
        Yo, ro, _ = oracle.qknorm_rms(workloads.bf16_bits(X), g.numpy(), eps, N)
        check_qk(workloads.bf16_bits(Y), r.cpu().numpy(), Yo, ro,
                 f"case {case}: T={T} H={N * W} N={N} eps={eps}")


def test_random_shapes_mx():
    rng = np.random.default_rng(20261203)
    for case in range(40):
        B = int(rng.choice([16, 32, 64]))
        fmt = "nvfp4" if B == 16 and rng.random() < 0.3 else str(rng.choice(["e4m3", "e2m1"]))
        D = B * int(rng.integers(1, max(2, 8192 // B)))
        T = int(rng.integers(1, 400))
        kind = str(rng.choice(["rms", "mx"]))
        p = int(rng.choice([1, 2]))
        with_gamma = bool(rng.random() < 0.5)
        X, g = workloads.mx_inputs(T, D, seed=2000 + case, t_frac=0.1, with_gamma=with_gamma)
        Xd = X.to(DEV)
        gd = None if g is None else g.to(DEV)
        if kind == "rms":
            out = nts.rmsnorm_mxcast(Xd, gd, B=B, fmt=fmt, want_rinv=True, want_amax=True)
            ref = oracle.rmsnorm_mxcast(workloads.bf16_bits(X), None if g is None else g.numpy(),
                                        1e-6, B, FMTS[fmt])
        else:
            out = nts.mxnorm_cast(Xd, gd, B=B, fmt=fmt, p=p, want_rinv=True, want_amax=True)
            ref = oracle.mxnorm_cast(workloads.bf16_bits(X), None if g is None else g.numpy(),
                                     1e-6, B, FMTS[fmt], p)
        nts.check_status()
        check_mx(workloads.bf16_bits(X), None if g is None else g.numpy(), B, FMTS[fmt],
                 (out.codes.cpu().numpy(), out.scales.cpu().numpy(), out.amax.cpu().numpy()),
                 ref, out.rinv.cpu().numpy(), 1e-6,
                 f"case {case}: {kind} p={p} T={T} D={D} B={B} {fmt} gamma={with_gamma}")

"""GPU parity of nts_rmsnorm_mxcast and nts_mxnorm_cast against the oracle,
through the C ABI.

Workloads: RMSNorm + MXFP8 cast vs MXNorm (p = 1, 2) on X [T, 4096] with
T in {4096, 16384, 65536}, B = 32, E4M3 (full size, sampled rows checked
against the oracle); the MXNorm sweep T = 65536, D in {1024, 3072, 5120, 7168,
16384}, B in {16, 32, 64}, E4M3 / E2M1, p = 2, 5% Student-t(3) rows (full
size on the device, sampled rows checked); small complete cases with gains;
edge cases (zero rows, tiny blocks, ragged tails, narrow rows, forced launch
shapes) and the bounded-wait error path.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_mx

pytestmark = pytest.mark.gpu

nts = pytest.importorskip("normalization_token_split_gb300")
DEV = "cuda:0"
FMTS = {"e4m3": oracle.FMT_E4M3, "e2m1": oracle.FMT_E2M1, "nvfp4": oracle.FMT_NVFP4}


def gpu_call(kind, X, gamma, eps, B, fmt, p):
    Xd = X.to(DEV)
    gd = None if gamma is None else gamma.to(DEV)
    if kind == "rms":
        out = nts.rmsnorm_mxcast(Xd, gd, eps=eps, B=B, fmt=fmt, want_rinv=True, want_amax=True)
    elif kind == "post":
        out = nts.mxnorm_postround_cast(Xd, gd, eps=eps, B=B, fmt=fmt, p=p, want_rinv=True,
                                        want_amax=True)
    else:
        out = nts.mxnorm_cast(Xd, gd, eps=eps, B=B, fmt=fmt, p=p, want_rinv=True, want_amax=True)
    nts.check_status()
    return out


def oracle_call(kind, Xb, g, eps, B, fmt, p):
    if kind == "rms":
        return oracle.rmsnorm_mxcast(Xb, g, eps, B, fmt)
    if kind == "post":
        return oracle.mxnorm_postround_cast(Xb, g, eps, B, fmt, p)
    return oracle.mxnorm_cast(Xb, g, eps, B, fmt, p)


def compare(kind, X, gamma, eps, B, fmt_name, p, rows=None, what=""):
    """Run the device; check all rows (rows=None) or the given sample."""
    fmt = FMTS[fmt_name]
    out = gpu_call(kind, X, gamma, eps, B, fmt_name, p)
    if rows is None:
        rows = slice(None)
    codes = out.codes[rows].cpu().numpy()
    scales = out.scales[rows].cpu().numpy()
    rinv = out.rinv[rows].cpu().numpy()
    amax = out.amax[rows].cpu().numpy()
    Xb = workloads.bf16_bits(X[rows])
    g = None if gamma is None else gamma.cpu().numpy()
    ref = oracle_call(kind, Xb, g, eps, B, fmt, p)
    return check_mx(Xb, g, B, fmt, (codes, scales, amax), ref, rinv, eps, what)


def sample_rows(T, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([rng.choice(T, size=min(n, T), replace=False),
                                     [0, T - 1]]))
    return torch.from_numpy(rows)


KINDS = [("rms", 0), ("mx", 1), ("mx", 2)]


@pytest.mark.parametrize("kind,p", KINDS)
@pytest.mark.parametrize("T", [4096, 16384, 65536])
def test_rmsnorm_mxcast_vs_mxnorm_config(kind, p, T):
    X, _ = workloads.mx_inputs(T, 4096, seed=4000 + T, device=DEV)
    rows = sample_rows(T, 2048, T).to(DEV)
    compare(kind, X, None, 1e-6, 32, "e4m3", p, rows=rows, what=f"{kind}{p} T={T}")


@pytest.mark.parametrize("D", [1024, 3072, 5120, 7168, 16384])
@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_mxnorm_sweep_full_size(D, B, fmt):
    X, _ = workloads.mx_inputs(65536, D, seed=5000 + D + B, t_frac=0.05, device=DEV)
    rows = sample_rows(65536, max(256, 4 * 1024 * 1024 // D), D + B)
    # heavy-tailed rows are part of the sample
    trows = torch.from_numpy(workloads.student_t_rows(65536, 5000 + D + B, 0.05)[:64])
    rows = torch.unique(torch.cat([rows, trows])).to(DEV)
    compare("mx", X, None, 1e-6, B, fmt, 2, rows=rows, what=f"sweep D={D} B={B} {fmt}")


@pytest.mark.parametrize("kind,p", KINDS)
@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("with_gamma", [False, True])
def test_small_complete(kind, p, B, fmt, with_gamma):
    X, g = workloads.mx_inputs(333, 1024, seed=B * 10 + p, t_frac=0.1, with_gamma=with_gamma)
    compare(kind, X, g, 1e-6, B, fmt, p, what=f"{kind}{p} B={B} {fmt} gamma={with_gamma}")


@pytest.mark.parametrize("D", [16, 32, 48, 64, 192, 1040, 2304, 8192, 32768])
@pytest.mark.parametrize("T", [1, 2, 5, 129])
def test_row_widths_and_ragged_tails(D, T):
    B = 16 if D % 32 else 32
    X, g = workloads.mx_inputs(T, D, seed=D + T, with_gamma=True)
    for kind, p in KINDS:
        for fmt in ("e4m3", "e2m1"):
            compare(kind, X, g, 1e-6, B, fmt, p, what=f"{kind}{p} T={T} D={D} {fmt}")


@pytest.mark.parametrize("B", [16, 32, 64])
def test_degenerate_blocks(B):
    X, _ = workloads.mx_inputs(64, 512, seed=77)
    X[0] = 0                          # all-zero row
    X[1, :B] = 0                      # one zero block
    X[5, B:3 * B] = 0                 # two zero blocks among ordinary ones
    X[2, 64:128] = 1e-38              # tiny blocks (scale clamps at 2^-127)
    X[3, 128:192] = -1.0e17           # large values (sum of squares stays finite in fp32)
    X[4, ::2] = -0.0
    X[6, 1::3] = 0                    # scattered zeros
    for kind, p in KINDS:
        for fmt in ("e4m3", "e2m1"):
            compare(kind, X, None, 1e-6, B, fmt, p, what=f"degenerate {kind}{p} B={B} {fmt}")


@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("with_gamma", [False, True])
def test_extreme_factors(B, with_gamma):
    # rows so small that the mean square underflows and rinv = 1/sqrt(eps)
    # is huge: rinv * 2^-e would overflow fp32 for some blocks, so a kernel
    # that folded the two products w*rinv and *2^-e into one would go wrong
    # there; fp32(w*rinv) itself is subnormal for some elements of others.
    # Ordinary rows share warps and tiles with them (both forms in one launch).
    X, g = workloads.mx_inputs(40, 1024, seed=78 + B, with_gamma=with_gamma)
    Xf = X.float()
    for r, sc in enumerate((1e-36, 1e-34, 1e-30, 1e-25, 1e-20, 1e-12, 3e-39, 1.0)):
        Xf[3 * r] *= sc
    X = Xf.to(torch.bfloat16)
    for kind, p in KINDS:
        for fmt in ("e4m3", "e2m1"):
            compare(kind, X, g, 1e-38, B, fmt, p,
                    what=f"extreme {kind}{p} B={B} {fmt} gamma={with_gamma}")


def test_zero_tokens_launches_nothing():
    X = torch.empty(0, 256, dtype=torch.bfloat16, device=DEV)
    out = nts.mxnorm_cast(X, None, B=32)
    nts.check_status()
    assert out.codes.shape == (0, 256) and out.scales.shape == (0, 8)


def test_deterministic():
    X, _ = workloads.mx_inputs(4096, 4096, seed=88, device=DEV)
    a = nts.mxnorm_cast(X, None, B=32, p=2, want_rinv=True)
    b = nts.mxnorm_cast(X, None, B=32, p=2, want_rinv=True)
    nts.check_status()
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    assert torch.equal(a.rinv, b.rinv)


@pytest.mark.parametrize("vpt,rows,stages,grid", [(1, 1, 1, 1), (2, 3, 2, 5), (3, 2, 4, 0),
                                                  (4, 4, 3, 7), (0, 0, 1, 0)])
def test_forced_launch_shapes(vpt, rows, stages, grid):
    X, g = workloads.mx_inputs(301, 2048, seed=99, with_gamma=True)
    try:
        nts.set_tuning(vpt=vpt, rows=rows, stages=stages, grid=grid)
        for kind, p in KINDS:
            compare(kind, X, g, 1e-6, 32, "e4m3", p, what=f"forced {vpt},{rows},{stages},{grid}")
    finally:
        nts.set_tuning()


@pytest.mark.parametrize("B,bpts", [(16, range(1, 9)), (32, range(1, 5)), (64, range(1, 5))])
def test_every_blocks_per_thread_count(B, bpts):
    # every instantiated blocks-per-thread count (half blocks for B = 64,
    # split between two lanes), on rows of 165 blocks of 16, 82 of 32 or 40
    # of 64 values, which most counts do not divide: the row's last thread
    # holds fewer units and its last warp idles in part
    D = 2640 if B == 16 else 2624 if B == 32 else 2560
    X, g = workloads.mx_inputs(150, D, seed=B + D, t_frac=0.1, with_gamma=True)
    try:
        for bpt in bpts:
            nts.set_tuning(vpt=bpt)
            for kind, p in KINDS:
                fmts = ("e4m3", "e2m1", "nvfp4") if B == 16 else ("e4m3", "e2m1")
                for fmt in fmts:
                    compare(kind, X, g, 1e-6, B, fmt, p, what=f"bpt={bpt} B={B} {kind}{p} {fmt}")
    finally:
        nts.set_tuning()


def test_blocks_per_thread_beyond_16_vectors_are_unsupported():
    X, _ = workloads.mx_inputs(64, 4096, seed=98, device=DEV)
    try:
        nts.set_tuning(vpt=5)             # 5 blocks of 32 = 20 vectors per thread
        with pytest.raises(nts.NtsError, match="UNSUPPORTED"):
            nts.mxnorm_cast(X, None, B=32, p=2)
    finally:
        nts.set_tuning()


@pytest.mark.parametrize("D,B", [(1024, 64), (512, 32), (256, 16), (128, 64)])
@pytest.mark.parametrize("T", [1, 3, 1000])
def test_half_warp_rows(D, B, T):
    # rows of at most 16 blocks take 16 threads: two rows per warp, each
    # summed over its own half of the warp
    X, g = workloads.mx_inputs(T, D, seed=D + B + T, t_frac=0.1, with_gamma=True)
    for kind, p in KINDS:
        for fmt in ("e4m3", "e2m1"):
            compare(kind, X, g, 1e-6, B, fmt, p, what=f"half-warp {kind}{p} D={D} B={B} T={T}")
            compare(kind, X, None, 1e-6, B, fmt, p, what=f"half-warp {kind}{p} D={D} B={B} T={T}")
    if B == 16:
        for kind, p in KINDS:
            if kind != "post":
                compare(kind, X, g, 1e-6, 16, "nvfp4", p, what=f"half-warp nvfp4 {kind}{p} D={D}")


def test_half_warp_rows_need_whole_warps():
    X, _ = workloads.mx_inputs(100, 1024, seed=97, device=DEV)
    try:
        nts.set_tuning(rows=3)            # 3 rows of 16 threads: not whole warps
        with pytest.raises(nts.NtsError, match="UNSUPPORTED"):
            nts.mxnorm_cast(X, None, B=64, p=2)
        nts.set_tuning(rows=6)
        a = nts.mxnorm_cast(X, None, B=64, p=2)
        nts.set_tuning()
        b = nts.mxnorm_cast(X, None, B=64, p=2)
        nts.check_status()
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    finally:
        nts.set_tuning()


def test_bounded_wait_reports_timeout_and_context_survives():
    X, _ = workloads.mx_inputs(64, 1024, seed=13)
    try:
        nts.set_wait_limit_ns(20_000_000)
        nts.set_missing_tx(16)
        nts.mxnorm_cast(X.to(DEV), None, B=32)
        with pytest.raises(nts.NtsError, match="TIMEOUT"):
            nts.check_status()
    finally:
        nts.set_missing_tx(0)
        nts.set_wait_limit_ns(0)
    compare("mx", X, None, 1e-6, 32, "e4m3", 2, what="after timeout")


@pytest.mark.parametrize("kind", ["rms", "mx"])
def test_host_buffer_form(kind):
    T, D, B = 700, 2048, 32
    X, _ = workloads.mx_inputs(T, D, seed=15)
    Xh = X.pin_memory()
    ch = torch.empty(T, D, dtype=torch.uint8).pin_memory()
    sh = torch.empty(T, D // B, dtype=torch.uint8).pin_memory()
    Xd = torch.empty_like(X, device=DEV)
    cd = torch.empty(T, D, dtype=torch.uint8, device=DEV)
    sd = torch.empty(T, D // B, dtype=torch.uint8, device=DEV)
    if kind == "rms":
        nts.rmsnorm_mxcast_host(Xh, None, ch, sh, Xd, cd, sd, eps=1e-6, B=B, fmt="e4m3")
    else:
        nts.mxnorm_cast_host(Xh, None, ch, sh, Xd, cd, sd, eps=1e-6, B=B, fmt="e4m3", p=2)
    nts.check_status()
    dev = gpu_call(kind, X, None, 1e-6, B, "e4m3", 2)
    assert torch.equal(ch, dev.codes.cpu()) and torch.equal(sh, dev.scales.cpu())


# ------------------------------------------------------ post-round MXNorm

@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("B", [16, 32, 64])
@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("with_gamma", [False, True])
def test_postround_small_complete(p, B, fmt, with_gamma):
    X, g = workloads.mx_inputs(257, 2048, seed=B * 3 + p, t_frac=0.1, with_gamma=with_gamma)
    compare("post", X, g, 1e-6, B, fmt, p, what=f"post p={p} B={B} {fmt} gamma={with_gamma}")


def test_postround_full_size_sampled():
    X, _ = workloads.mx_inputs(65536, 4096, seed=4100, device=DEV)
    rows = sample_rows(65536, 2048, 7).to(DEV)
    for p in (1, 2):
        compare("post", X, None, 1e-6, 32, "e4m3", p, rows=rows, what=f"post full p={p}")


def test_postround_subnormal_and_degenerate_blocks():
    X, _ = workloads.mx_inputs(32, 512, seed=43)
    X[0] = 0
    X[1, :32] = 3.0e-39                # bf16 subnormal block absmax
    X[2, 32:64] = 7.0e-40
    X[3] = 2.0e-38                     # a whole row of tiny values
    X[4, ::2] = -0.0
    for p in (1, 2):
        for fmt in ("e4m3", "e2m1"):
            compare("post", X, None, 1e-6, 32, fmt, p, what=f"post degenerate p={p} {fmt}")


# ------------------------------------------- NVFP4 (E2M1, B = 16, E4M3 scales)

@pytest.mark.parametrize("kind,p", KINDS)
@pytest.mark.parametrize("with_gamma", [False, True])
def test_nvfp4_small_complete(kind, p, with_gamma):
    X, g = workloads.mx_inputs(333, 1024, seed=900 + p, t_frac=0.1, with_gamma=with_gamma)
    compare(kind, X, g, 1e-6, 16, "nvfp4", p, what=f"nvfp4 {kind}{p} gamma={with_gamma}")


@pytest.mark.parametrize("kind,p", KINDS)
@pytest.mark.parametrize("D", [4096, 7168, 16384])
def test_nvfp4_full_size_sampled(kind, p, D):
    X, _ = workloads.mx_inputs(65536, D, seed=910 + D, t_frac=0.05, device=DEV)
    rows = sample_rows(65536, max(256, 4 * 1024 * 1024 // D), D + p)
    trows = torch.from_numpy(workloads.student_t_rows(65536, 910 + D, 0.05)[:64])
    rows = torch.unique(torch.cat([rows, trows])).to(DEV)
    compare(kind, X, None, 1e-6, 16, "nvfp4", p, rows=rows, what=f"nvfp4 {kind}{p} D={D}")


@pytest.mark.parametrize("D", [16, 48, 1040, 8192, 32768])
@pytest.mark.parametrize("T", [1, 5, 129])
def test_nvfp4_row_widths_and_ragged_tails(D, T):
    X, g = workloads.mx_inputs(T, D, seed=920 + D + T, with_gamma=True)
    for kind, p in KINDS:
        compare(kind, X, g, 1e-6, 16, "nvfp4", p, what=f"nvfp4 {kind}{p} T={T} D={D}")


def test_nvfp4_degenerate_blocks():
    X, _ = workloads.mx_inputs(64, 512, seed=930)
    X[0] = 0                          # all-zero row: zero scales and codes
    X[1, :16] = 0                     # one zero block
    X[2, 32:48] = 1e-30               # block whose scale underflows to zero
    X[3, 64:80] = -1.0e17             # large values
    X[4, ::2] = -0.0
    X[5, 96:112] = torch.linspace(-3, 3, 16)
    for kind, p in KINDS:
        out = gpu_call(kind, X, None, 1e-6, 16, "nvfp4", p)
        compare(kind, X, None, 1e-6, 16, "nvfp4", p, what=f"nvfp4 degenerate {kind}{p}")
        sc = out.scales.cpu().numpy()
        assert np.all(sc[0] == 0) and sc[1, 0] == 0 and sc[2, 2] == 0
        assert np.all(out.codes[0].cpu().numpy() == 0)
        assert np.all(out.codes[2, 16:24].cpu().numpy() == 0)


def test_nvfp4_rejects_other_blocks_and_post_round():
    X, _ = workloads.mx_inputs(4, 256, seed=931, device=DEV)
    with pytest.raises(nts.NtsError, match="INVALID_ARG"):
        nts.rmsnorm_mxcast(X, None, B=32, fmt="nvfp4")
    with pytest.raises(nts.NtsError, match="INVALID_ARG"):
        nts.mxnorm_postround_cast(X, None, B=16, fmt="nvfp4")


def test_nvfp4_scale_without_division_matches_ieee_route():
    # Every non-negative fp32 absmax, 0 to +inf, on the device: the kernels'
    # scale code and reciprocal (division by 6 without a divide, reciprocal
    # from a table) equal those through the IEEE quotient and reciprocal, and
    # the division is the IEEE quotient wherever that quotient is normal.
    code_bad, quot_bad = nts.check_nvfp4_scale()
    assert code_bad == 0, f"{code_bad} absmaxes with another scale or reciprocal"
    assert quot_bad == 0, f"{quot_bad} normal quotients differ from IEEE division"


def test_e8m0_exponent_by_carry_matches_definition():
    # every non-negative fp32 absmax, 0 to +inf, for E4M3 and E2M1: the
    # kernels' one-add exponent equals the field-by-field definition
    assert nts.check_e8m0() == 0


# ------------------------------------------------------------ tile order

def test_dynamic_and_round_robin_tile_orders_agree():
    # tiles taken from the per-stream counter or round-robin: same results,
    # and the counter re-arms itself between back-to-back launches
    X, _ = workloads.mx_inputs(5003, 2048, seed=950, t_frac=0.05, device=DEV)
    outs = []
    try:
        for dyn in (True, False, True):
            nts.set_schedule(dyn)
            for _ in range(3):
                out = nts.mxnorm_cast(X, None, B=32, p=2, want_rinv=True)
            nts.check_status()
            outs.append(out)
    finally:
        nts.set_schedule(True)
    for o in outs[1:]:
        assert torch.equal(o.codes, outs[0].codes) and torch.equal(o.scales, outs[0].scales)
        assert torch.equal(o.rinv, outs[0].rinv)


def test_launches_on_several_streams():
    # each stream owns its counter pair: overlapping launches do not share one
    Xs = [workloads.mx_inputs(T, 1024, seed=960 + T, device=DEV)[0] for T in (3001, 777, 4096)]
    want = [nts.rmsnorm_mxcast(X, None, B=32) for X in Xs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in Xs]
    got = [[None] * 4 for _ in Xs]
    for rep in range(4):
        for i, (X, st) in enumerate(zip(Xs, streams)):
            with torch.cuda.stream(st):
                got[i][rep] = nts.rmsnorm_mxcast(X, None, B=32, stream=st)
    torch.cuda.synchronize()
    nts.check_status()
    for w, gs in zip(want, got):
        for g in gs:
            assert torch.equal(g.codes, w.codes) and torch.equal(g.scales, w.scales)


@pytest.mark.parametrize("T,D,B,fmt", [(20011, 4096, 32, "e4m3"), (9000, 2048, 16, "nvfp4"),
                                       (4133, 8192, 32, "e2m1")])
def test_host_buffer_form_in_chunks(T, D, B, fmt):
    # large enough to be split into chunks that flow through the copy-in,
    # kernel and copy-out streams; the last chunk is ragged
    X, _ = workloads.mx_inputs(T, D, seed=16 + T, t_frac=0.05)
    Xh = X.pin_memory()
    cb = D if fmt == "e4m3" else D // 2
    ch = torch.empty(T, cb, dtype=torch.uint8).pin_memory()
    sh = torch.empty(T, D // B, dtype=torch.uint8).pin_memory()
    Xd = torch.empty_like(X, device=DEV)
    cd = torch.empty(T, cb, dtype=torch.uint8, device=DEV)
    sd = torch.empty(T, D // B, dtype=torch.uint8, device=DEV)
    for rep in range(2):
        nts.mxnorm_cast_host(Xh, None, ch, sh, Xd, cd, sd, eps=1e-6, B=B, fmt=fmt, p=2)
        nts.check_status()
        dev = nts.mxnorm_cast(X.to(DEV), None, eps=1e-6, B=B, fmt=fmt, p=2)
        nts.check_status()
        assert torch.equal(ch, dev.codes.cpu()) and torch.equal(sh, dev.scales.cpu())
        ch.zero_()


@pytest.mark.parametrize("chunks,min_bytes", [(64, 1 << 20), (7, 1 << 20), (2, 1 << 20), (1, 0)])
def test_host_buffer_form_any_chunking(chunks, min_bytes):
    # the chunk count changes only how the rows flow through the copy
    # streams: the outputs are those of the device path bit for bit
    T, D = 7001, 2048
    X, _ = workloads.mx_inputs(T, D, seed=17 + chunks, t_frac=0.05)
    Xh = X.pin_memory()
    ch = torch.empty(T, D // 2, dtype=torch.uint8).pin_memory()
    sh = torch.empty(T, D // 32, dtype=torch.uint8).pin_memory()
    Xd = torch.empty_like(X, device=DEV)
    cd = torch.empty(T, D // 2, dtype=torch.uint8, device=DEV)
    sd = torch.empty(T, D // 32, dtype=torch.uint8, device=DEV)
    try:
        nts.set_host_chunks(chunks, min_bytes)
        nts.rmsnorm_mxcast_host(Xh, None, ch, sh, Xd, cd, sd, eps=1e-6, B=32, fmt="e2m1")
        nts.check_status()
    finally:
        nts.set_host_chunks()
    ref = nts.rmsnorm_mxcast(X.to(DEV), None, eps=1e-6, B=32, fmt="e2m1")
    nts.check_status()
    assert torch.equal(ch, ref.codes.cpu()) and torch.equal(sh, ref.scales.cpu())


def test_graph_replays_alongside_direct_launches():
    # a launch recorded into a CUDA graph owns its tile counters; direct
    # launches on other streams keep theirs, so the two never share one.  The
    # graph clears its outputs first, so a replay whose counters were not
    # re-armed by the previous one would leave zeros behind.
    X1, _ = workloads.mx_inputs(6000, 2048, seed=980, device=DEV)
    X2, _ = workloads.mx_inputs(7000, 2048, seed=981, device=DEV)
    ref1 = nts.mxnorm_cast(X1, None, B=32, p=2)
    ref2 = nts.mxnorm_cast(X2, None, B=32, p=2)
    c1 = torch.empty_like(ref1.codes)
    s1 = torch.empty_like(ref1.scales)
    c1b = torch.empty_like(ref1.codes)
    s1b = torch.empty_like(ref1.scales)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        c1.zero_()
        s1.zero_()
        nts.mxnorm_cast(X1, None, B=32, p=2, codes=c1, scales=s1)
        c1b.zero_()
        s1b.zero_()
        nts.mxnorm_cast(X1, None, B=32, p=2, codes=c1b, scales=s1b)   # a second node
    side = torch.cuda.Stream()
    outs = []
    for _ in range(6):
        graph.replay()
        with torch.cuda.stream(side):
            outs.append(nts.mxnorm_cast(X2, None, B=32, p=2, stream=side))
        torch.cuda.current_stream().synchronize()
        assert torch.equal(c1, ref1.codes) and torch.equal(s1, ref1.scales)
        assert torch.equal(c1b, ref1.codes) and torch.equal(s1b, ref1.scales)
    torch.cuda.synchronize()
    nts.check_status()
    for o in outs:
        assert torch.equal(o.codes, ref2.codes) and torch.equal(o.scales, ref2.scales)


def test_graphs_replayed_on_two_streams_at_once():
    # two captured graphs (each with its own counters) replayed concurrently
    # on two streams, many times, with the QK kernel's counters in use too
    X, _ = workloads.mx_inputs(9000, 4096, seed=982, device=DEV)
    Q, gq = workloads.qk_inputs(3000, 5120, seed=983, device=DEV)
    refm = nts.rmsnorm_mxcast(X, None, B=32)
    refq, _ = nts.qknorm_rms(Q, gq, N=4)
    cm, sm = torch.empty_like(refm.codes), torch.empty_like(refm.scales)
    yq = torch.empty_like(refq)
    torch.cuda.synchronize()
    g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1):
        cm.zero_()
        nts.rmsnorm_mxcast(X, None, B=32, codes=cm, scales=sm)
    with torch.cuda.graph(g2):
        yq.zero_()
        nts.qknorm_rms(Q, gq, N=4, out=yq)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(5):
        with torch.cuda.stream(s1):
            g1.replay()
        with torch.cuda.stream(s2):
            g2.replay()
        torch.cuda.synchronize()
        assert torch.equal(cm, refm.codes) and torch.equal(sm, refm.scales)
        assert torch.equal(yq, refq)
    nts.check_status()


def test_boundary_exception_counts_are_a_handful(capsys):
    # The double-precision definition and the kernel's fp32 decisions may
    # differ only where a value sits within 1e-6 of a rounding boundary;
    # count those exceptions over every row of the 65536 x 4096 config.
    X, _ = workloads.mx_inputs(65536, 4096, seed=4000 + 65536, device=DEV)
    report = {}
    for kind, p in KINDS:
        totals = {"scale_boundary_exceptions": 0, "code_boundary_exceptions": 0}
        for r0 in range(0, 65536, 8192):
            rows = torch.arange(r0, r0 + 8192, device=DEV)
            st = compare(kind, X, None, 1e-6, 32, "e4m3", p, rows=rows, what=f"{kind}{p}")
            for k in totals:
                totals[k] += st[k]
        report[f"{kind}{p}"] = totals
        blocks = 65536 * 128
        assert totals["scale_boundary_exceptions"] <= blocks * 1e-4
        assert totals["code_boundary_exceptions"] <= blocks * 32 * 1e-5
    with capsys.disabled():
        print("\nMX boundary exceptions over 65536 x 4096 (B=32, E4M3):", report)

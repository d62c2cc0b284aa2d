"""The MX launch rules, checked on the host over a wide grid of requests
(nts_debug_mx_launch_shape computes the shape launch_mx would use, without
a device): every shape must satisfy what the kernel assumes.

* a row takes 16 threads (two rows per warp) or whole warps, and a tile
  whole warps, at most 480 consumer threads;
* the row's units (blocks; halves of 64-value blocks) are covered:
  threads * units per thread >= units, with at most 16 vectors per thread;
* 64-value blocks are split between lane pairs: an even unit count and an
  even thread count per row;
* the ring of at least one stage fits the device's opt-in shared memory,
  and its size is the layout's: stages * rows * D * 2 bytes plus barriers;
* a tile of rows at least 8 KB or four warps when T allows, fewer rows
  only when T is small.
"""
import ctypes
import itertools

import pytest

nts = pytest.importorskip("normalization_token_split_gb300")
from normalization_token_split_gb300 import _lib  # noqa: E402

E4M3, E2M1, NVFP4 = 0, 1, 2
SM, SMEM = 152, 232448          # GB300: SMs and opt-in shared memory per CTA
INVALID, UNSUPPORTED, OK = 1, 2, 0


def shape(T, D, B, fmt, p=2, sm=SM, smem=SMEM, regs=96):
    out = (ctypes.c_int32 * 5)()
    rc = _lib.lib().nts_debug_mx_launch_shape(T, D, B, fmt, p, sm, smem, regs, out)
    return rc, list(out)


def ctas_per_sm(threads, smem_cta, regs, smem_optin=SMEM):
    """CTAs per SM on GB300: 228 KB of shared memory with 1 KB reserved per
    CTA, 64 K registers allocated per warp in units of 8 per thread, 2048
    threads."""
    warps = -(-threads // 32)
    n = (smem_optin + 1024) // (smem_cta + 1024)
    if regs:
        n = min(n, 65536 // (-(-regs // 8) * 8 * 32 * warps))
    return min(n, 2048 // (warps * 32), 32)


def widths():
    ds = set(range(16, 4097, 16)) | set(range(4096, 32769, 1024)) | {1040, 2640, 5120, 7168}
    return sorted(ds)


@pytest.mark.parametrize("B", [16, 32, 64])
def test_every_shape_satisfies_the_kernel(B):
    fmts = [E4M3, E2M1] + ([NVFP4] if B == 16 else [])
    checked = 0
    for D, T, fmt in itertools.product(widths(), [1, 5, 300, 4097, 65536], fmts):
        if D % B:
            continue
        rc, (bpt, G, R, S, smem) = shape(T, D, B, fmt)
        if rc != OK:
            # only rows too wide for shared memory may be refused
            assert rc == UNSUPPORTED and D * 2 > SMEM // 2, (D, B, T, fmt, rc)
            continue
        checked += 1
        what = f"D={D} B={B} T={T} fmt={fmt}: bpt={bpt} G={G} R={R} S={S}"
        unit_vectors = 4 if B == 64 else B // 8
        units = 2 * (D // B) if B == 64 else D // B
        assert G == 16 or G % 32 == 0, what
        assert (R * G) % 32 == 0 and R * G <= 480, what
        assert G * bpt >= units and bpt * unit_vectors <= 16, what
        n = -(-units // bpt)                               # threads that hold units
        assert G == (16 if n <= 16 else -(-n // 32) * 32), what   # no idle warp
        if B == 64:
            assert units % 2 == 0 and G % 2 == 0, what
        assert S >= 1 and smem <= SMEM, what
        assert smem >= S * R * D * 2, what
        if T >= 2 * SM * 16:
            assert R * D * 2 >= 8192 or R * G >= 128 or R * G + G > 480, what
    assert checked > 500


def test_small_token_counts_spread_rows_over_the_gpu():
    # rows per tile shrink until every SM gets at least two tiles, but never
    # below whole warps
    for D, B in ((4096, 32), (1024, 64), (256, 16)):
        _, (_, G, R_big, _, _) = shape(65536, D, B, E4M3)
        _, (_, G2, R_small, _, _) = shape(100, D, B, E4M3)
        assert G == G2 and R_small <= R_big and (R_small * G2) % 32 == 0


def test_measured_shapes():
    # the shapes the measurements chose (DESIGN: MX mapping)
    assert shape(65536, 4096, 32, E4M3)[1][:2] == [4, 32]
    assert shape(65536, 5120, 32, E4M3)[1][:2] == [3, 64]
    assert shape(65536, 5120, 16, E4M3)[1][:2] == [5, 64]
    assert shape(65536, 7168, 16, E2M1)[1][:2] == [7, 64]
    assert shape(65536, 1024, 64, E4M3)[1][:2] == [2, 16]     # 32 half blocks on 16 threads
    assert shape(65536, 3072, 32, E4M3)[1][:2] == [3, 32]
    # two stages for rows above 24 KB a stage (three CTAs per SM)
    assert shape(65536, 7168, 32, E4M3)[1][3] == 2
    # the ring depth keeps the most CTAs per SM: two stages of two 10 KB rows
    # at D = 5120 (four CTAs of 96 registers per thread, where three stages
    # leave three), three stages of 16 KB at D = 1024 (four CTAs either way)
    assert shape(65536, 5120, 16, E2M1)[1][2:4] == [2, 2]
    assert shape(65536, 3072, 32, E4M3)[1][3] == 2
    assert shape(65536, 1024, 16, E2M1)[1][2:4] == [8, 3]
    # with 104 registers only three CTAs fit anyway: the deeper ring
    assert shape(65536, 3072, 32, E4M3, regs=104)[1][3] == 3


@pytest.mark.parametrize("regs", [0, 64, 96, 104, 128])
def test_ring_depth_keeps_the_most_ctas_per_sm(regs):
    # over the grid of widths: the chosen ring holds as many CTAs per SM as
    # two stages would, and no deeper ring of at most four stages does
    for D, B in itertools.product(widths(), [16, 32, 64]):
        if D % B:
            continue
        rc, (bpt, G, R, S, smem) = shape(65536, D, B, E4M3, regs=regs)
        if rc != OK or S < 2:
            continue
        threads = R * G + 32
        stage = R * D * 2
        fixed = smem - S * stage                     # barriers and slots
        best = ctas_per_sm(threads, fixed + 2 * stage, regs)
        assert ctas_per_sm(threads, smem, regs) == best, (D, B, regs, R, S)
        for deeper in range(S + 1, 5):
            size = fixed + deeper * stage
            assert size > 102400 or ctas_per_sm(threads, size, regs) < best, (D, B, regs, S)


def test_query_arguments():
    out = (ctypes.c_int32 * 5)()
    lib = _lib.lib()
    assert lib.nts_debug_mx_launch_shape(10, 100, 32, E4M3, 2, SM, SMEM, 96, out) == INVALID  # D % B
    assert lib.nts_debug_mx_launch_shape(10, 256, 32, NVFP4, 2, SM, SMEM, 96, out) == INVALID
    assert lib.nts_debug_mx_launch_shape(10, 256, 32, E4M3, 3, SM, SMEM, 96, out) == INVALID
    assert lib.nts_debug_mx_launch_shape(10, 256, 32, E4M3, 2, SM, SMEM, 96, None) == INVALID
    assert lib.nts_debug_mx_launch_shape(10, 256, 32, E4M3, 2, SM, SMEM, -1, out) == INVALID
    assert lib.nts_debug_mx_launch_shape(10, 256, 32, E4M3, 2, SM, SMEM, 256, out) == INVALID
    assert lib.nts_debug_mx_launch_shape(10, 256, 32, E4M3, 2, SM, SMEM, 96, out) == OK

"""The NVFP4 block scale divides the normalized absmax by 6 without a divide
instruction: q = fl(a z) with z = fl(1/6), the remainder r = a - 6q exact in
one fma, then fl(q + r z) (Brisebarre, Muller and Raina, "Accelerating
correctly rounded floating-point division when the divisor is known in
advance", IEEE Trans. Computers 53(8), 2004).  The CUDA kernels rely on this
being the IEEE quotient wherever the quotient is a normal fp32.

While q and the quotient are normal, r = a - 6q is an exact fp32 and every
step scales exactly with a by powers of two, so one binade of a decides all
binades but those next to the underflow threshold and to the overflow end.  This test runs, in C with
the host's correctly rounded fmaf, every a of the binade [1, 2), every a of
the binades around 6 * 2^-126 (where the quotient becomes subnormal) and the
top binade of fp32, and compares with IEEE division.  The device-side check
over every fp32 value is test_gpu_mx.py's.
"""
import os
import shutil
import subprocess

import pytest

C_SOURCE = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }
static uint32_t to_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }

/* a from bit patterns lo .. hi-1; counts the quotients >= 2^-126 that differ */
static unsigned long long run(uint32_t lo, uint32_t hi) {
    volatile float z = 1.0f / 6.0f;     /* fl(1/6) */
    unsigned long long bad = 0;
    for (uint32_t u = lo; u < hi; ++u) {
        float a = from_bits(u);
        float q = a * z;
        float r = fmaf(-q, 6.0f, a);
        float d = fmaf(r, z, q);
        float ieee = a / 6.0f;
        if (ieee >= 0x1p-126f && to_bits(d) != to_bits(ieee)) ++bad;
    }
    return bad;
}

int main(void) {
    unsigned long long bad = 0;
    bad += run(0x3F800000u, 0x40000000u);   /* [1, 2) */
    bad += run(0x00800000u, 0x02000000u);   /* [2^-126, 2^-123): quotients near 2^-126 */
    bad += run(0x7F000000u, 0x7F800000u);   /* [2^127, max] */
    printf("%llu %a\n", bad, (double)(1.0f / 6.0f));
    return 0;
}
"""


def test_division_by_six_is_the_ieee_quotient(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "div6.c"
    exe = tmp_path / "div6"
    src.write_text(C_SOURCE)
    # -ffp-contract=off: the multiply must not fuse with anything
    subprocess.run([cc, "-O1", "-ffp-contract=off", "-fno-fast-math", "-o", str(exe), str(src),
                    "-lm"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True,
                         timeout=600).stdout.split()
    assert out[1] == "0x1.555556p-3"          # z = fl(1/6) is the constant the kernels use
    assert int(out[0]) == 0

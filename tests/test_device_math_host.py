"""Host checks of arithmetic identities the kernels rely on (CPU only).

The double block's outer scale s_o = amax / 2688 must be the IEEE quotient
("Resumo Técnico: TetraJet-v2", §2A: an FP32 scale per 1x128 block).  The
kernels compute it without a division: q0 = amax * R with R = RN(1 / 2688),
then q = fma(fma(-q0, 2688, amax), R, q0), and fall back to the division for
amax < 2^-119.  Both steps are single IEEE operations with round-to-nearest,
which C's `*` and `fmaf` reproduce on the host, so the identity is checked
here against C's division: over every FP32 pattern of [2^-119, FLT_MAX] with
a stride of 3 (all exponents, a third of the mantissas; the full sweep was
also run once, with no mismatch), and the constant R itself.

Stochastic rounding treats |y| < 1 on the grid of [1, 2) (it adds 1 first),
and selects that case with q = sat(fma(|y|, -2^24, 2^24)) (a saturating FMA,
clamped to [0, 1], NaN to 0) rather than a comparison.  That q is 1 exactly
when |y| < 1 and 0 otherwise is checked over every non-negative FP32 pattern,
infinities and NaNs included.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

SRC = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <math.h>
static float f(uint32_t b) { float x; memcpy(&x, &b, 4); return x; }
static uint32_t u(float x) { uint32_t b; memcpy(&b, &x, 4); return b; }
int main(void)
{
    const float D = 2688.0f;
    volatile float one = 1.0f;
    const float R = 0x1.861862p-12f;
    if (u(one / D) != u(R)) { printf("R mismatch\n"); return 2; }
    const uint32_t lo = u(0x1p-119f);
    unsigned long long bad = 0, n = 0;
    for (uint32_t b = lo; b < 0x7F800000u; b += 3) {
        float x = f(b);
        float q0 = x * R;
        float q = fmaf(fmaf(-q0, D, x), R, q0);
        n++;
        if (u(q) != u(x / D)) bad++;
    }
    printf("%llu %llu\n", n, bad);
    return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_outer_scale_division_free_form_equals_ieee_division():
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "chk.c")
        exe = os.path.join(d, "chk")
        with open(c, "w") as fh:
            fh.write(SRC)
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe, c, "-lm"],
                       check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout
    n, bad = map(int, r.stdout.split())
    assert bad == 0 and n > 600_000_000


SRC_SEL = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <math.h>
static float f(uint32_t b) { float x; memcpy(&x, &b, 4); return x; }
int main(void)
{
    unsigned long long bad = 0, n = 0;
    for (uint64_t b = 0; b <= 0x7FFFFFFFu; ++b) {
        const float a = f((uint32_t)b);
        const float r = fmaf(a, -0x1p24f, 0x1p24f);
        const float q = r > 0.0f ? (r < 1.0f ? r : 1.0f) : 0.0f;  /* .sat: NaN -> 0 */
        const float want = a < 1.0f ? 1.0f : 0.0f;
        n++;
        if (q != want) bad++;
    }
    printf("%llu %llu\n", n, bad);
    return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_sr_below_one_selector_by_saturating_fma():
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "sel.c")
        exe = os.path.join(d, "sel")
        with open(c, "w") as fh:
            fh.write(SRC_SEL)
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe, c, "-lm"],
                       check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout
    n, bad = map(int, r.stdout.split())
    assert bad == 0 and n == 2 ** 31

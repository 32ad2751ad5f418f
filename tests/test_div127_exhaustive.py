"""The quantizer's division-free scale: d = amax/127 as q0 = amax*r, then q0 + r*(amax - 127*q0) with r the
rounded 1/127 and the residual and the correction each one fused multiply-add (Markstein's correction step),
must equal the correctly rounded IEEE quotient amax/127 for every non-negative finite f32 amax (2^31 - 2^23
values, zero and subnormals included).  The check is plain C on the host: f32 products, fmaf and the
division are all IEEE round-to-nearest there as on the GPU (no fast-math, subnormals kept)."""
import os
import subprocess
import tempfile

import pytest

C_SRC = r"""
#include <stdio.h>
#include <stdint.h>
#include <string.h>
#include <math.h>
int main(void) {
    const float y = 127.0f, r = 1.0f / 127.0f;
    unsigned long long bad = 0;
    for (uint64_t u = 0; u < 0x7f800000ull; u++) {
        float a; uint32_t ui = (uint32_t)u; memcpy(&a, &ui, 4);
        const float want = a / y;
        const float q0 = a * r;
        const float got = fmaf(fmaf(-q0, y, a), r, q0);
        uint32_t bw, bg; memcpy(&bw, &want, 4); memcpy(&bg, &got, 4);
        bad += bw != bg;
    }
    printf("%llu\n", bad);
    return 0;
}
"""


@pytest.mark.timeout(600)
def test_division_free_scale_equals_ieee_quotient_for_every_amax():
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "div127.c"), os.path.join(d, "div127")
        with open(src, "w") as f:
            f.write(C_SRC)
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe, src, "-lm"], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.strip()
    assert out == "0"

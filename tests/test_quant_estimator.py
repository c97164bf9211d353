"""The quantizer's fast code estimate, checked on every fp32 quotient (CPU).

nf4_quantize decides most codes from q = w * rcp(absmax) with a degree-5
polynomial h: est = round(h(q)), then code = est + (q > T[est]).  That is
right only if est is the code of q or one below it, for every fp32 q the
kernel can see (|q| <= 1 + a few ulps).  This test reads the polynomial's
constants from the CUDA source, takes the thresholds from the published
codebook (tests/golden/nf4_codebook.txt, exact fp64 midpoints rounded down to
fp32: the tie rule "nearest, ties to the lower index"), and walks all 2.1e9
fp32 values in [-1 - 8 ulp, 1 + 8 ulp] in a small C program: h is evaluated
in double precision and must stay at least 1e-3 inside the interval where
rounding gives code - 1 or code, far more than the kernel's fp32 Horner
error (< 1e-5 for |h| <= 16).  This is a check of the kernel's arithmetic
from the kernel's own constants; the oracle is not involved.
"""
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
QUANT_CU = os.path.join(ROOT, "nf4_weight_quantized_quantize_gb300", "csrc", "nf4_quant.cu")
CODEBOOK = os.path.join(ROOT, "tests", "golden", "nf4_codebook.txt")

CHECKER = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static float f_of(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
int main(int argc, char** argv) {
    (void)argc;
    double c[6]; float t[15];
    for (int i = 0; i < 6; ++i) c[i] = (double)(float)strtod_wrap(argv[1 + i]);
    for (int j = 0; j < 15; ++j) t[j] = (float)strtod_wrap(argv[7 + j]);
    const double margin = 1e-3;
    const uint32_t hi = 0x3f800008u;   /* 1 + 8 ulp */
    long long bad = 0, n = 0;
    double worst = 1e9;
    #pragma omp parallel for reduction(+:bad,n) reduction(min:worst) schedule(static)
    for (long long k = 0; k <= 2LL * hi + 1; ++k) {
        const uint32_t b = (uint32_t)(k >> 1);
        const float q = (k & 1) ? -f_of(b) : f_of(b);
        int code = 0;
        for (int j = 0; j < 15; ++j) code += q > t[j];
        const double x = (double)q;
        const double h = ((((c[0] * x + c[1]) * x + c[2]) * x + c[3]) * x + c[4]) * x + c[5];
        const double lo_gap = h - ((double)code - 1.5), hi_gap = ((double)code + 0.5) - h;
        const double g = lo_gap < hi_gap ? lo_gap : hi_gap;
        if (g < worst) worst = g;
        /* round(h) must also index the 16-entry table */
        if (g < margin || h < -0.5 + margin || h > 15.5 - margin) ++bad;
        ++n;
    }
    printf("%lld %lld %.6f\n", n, bad, worst);
    return 0;
}
"""


def kernel_constants():
    text = open(QUANT_CU).read()
    vals = {}
    for name in ("kH5", "kH4", "kH3", "kH2", "kH1", "kH0Magic"):
        m = re.search(rf"constexpr float {name} = ([-0-9.eE+]+)f;", text)
        assert m, f"{name} not found in nf4_quant.cu"
        vals[name] = float(m.group(1))
    magic = float(np.float32(1.5 * 2 ** 23))
    c0 = float(np.float32(vals["kH0Magic"])) - magic
    assert c0 == round(c0), "the constant term must be an integer so the rounding can ride on the last FMA"
    return [vals["kH5"], vals["kH4"], vals["kH3"], vals["kH2"], vals["kH1"], c0]


def thresholds():
    cb = [float(v) for v in open(CODEBOOK).read().split("\n") if v.strip() and not v.startswith("#")]
    c = np.array(cb, dtype=np.float32).astype(np.float64)
    mid = (c[:-1] + c[1:]) / 2
    t = mid.astype(np.float32)
    t = np.where(t.astype(np.float64) > mid, np.nextafter(t, np.float32(-2)), t).astype(np.float32)
    assert (t.astype(np.float64) <= mid).all()
    return [float(v) for v in t]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_estimate_is_code_or_one_below_for_every_fp32_quotient(tmp_path):
    src = tmp_path / "est_check.c"
    src.write_text("#include <stdlib.h>\nstatic double strtod_wrap(const char* s) { return strtod(s, 0); }\n"
                   + CHECKER)
    exe = tmp_path / "est_check"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", str(src), "-o", str(exe)],
                   check=True)
    args = [repr(float(np.float32(v))) for v in kernel_constants()] + [repr(v) for v in thresholds()]
    out = subprocess.run([str(exe), *args], check=True, capture_output=True, text=True, timeout=600).stdout
    n, bad, worst = out.split()
    assert int(n) == 2 * (0x3F800008 + 1)
    assert int(bad) == 0, f"{bad} quotients where round(h(q)) is not code or code - 1 (worst margin {worst})"
    assert float(worst) > 1e-3

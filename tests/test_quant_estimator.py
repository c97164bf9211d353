"""The quantizer's fast code selection, checked on every fp32 quotient (CPU).

nf4_quantize decides most codes from q = w * rcp(absmax) through a cell table:
cell c = round(16 q + 16) (the fp32 sum 16 q + 16 + 1.5 * 2^23, whose low
mantissa bits hold c), entry e = table[c & 63] -- a threshold with its low four
fraction bits replaced by its index + 1 -- and code = (bits(e) & 15) - 1 +
(q > e).  The kernel takes that code only when |q - e| > guard and redoes the
word by exact division otherwise.  This test reads the table, the cell
constant and the guard from the CUDA source, takes the thresholds from the
published codebook (tests/golden/nf4_codebook.txt, exact fp64 midpoints
rounded down to fp32: the tie rule "nearest, ties to the lower index"), and
walks all 2.1e9 fp32 values in [-1 - 8 ulp, 1 + 8 ulp] in a small C program,
with the kernel's fp32 roundings.  Wherever the fast path is taken its code
must be the code of q, and every threshold must be more than 2^-21 from q --
farther than the exact quotient n = w / absmax can be from q (|q - n| <=
3 * 2^-24 |n|), so n has the same code.  The cell index must stay in 0 .. 32.
A check of the kernel's arithmetic from the kernel's own constants; the oracle
is not involved.
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
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
static float f_of(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t b_of(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }
int main(int argc, char** argv) {
    (void)argc;
    uint32_t cell[64]; float t[15];
    const float magic = strtof(argv[1], 0), guard = strtof(argv[2], 0);
    for (int i = 0; i < 64; ++i) cell[i] = (uint32_t)strtoul(argv[3 + i], 0, 0);
    for (int j = 0; j < 15; ++j) t[j] = strtof(argv[67 + j], 0);
    const uint32_t hi = 0x3f800008u;   /* 1 + 8 ulp */
    long long n = 0, wrong = 0, near = 0, slow = 0, badidx = 0;
    #pragma omp parallel for reduction(+:n,wrong,near,slow,badidx) schedule(static)
    for (long long k = 0; k <= 2LL * hi + 1; ++k) {
        const uint32_t b = (uint32_t)(k >> 1);
        const float q = (k & 1) ? -f_of(b) : f_of(b);
        int code = 0;
        for (int j = 0; j < 15; ++j) code += q > t[j];
        const float cm = q * 16.0f + magic;            /* 16 q exact, one rounding */
        const uint32_t idx = b_of(cm) & 63u;
        if (idx > 32u) ++badidx;
        const uint32_t e = cell[idx];
        const float d = q - f_of(e);
        ++n;
        if (!(fabsf(d) > guard)) { ++slow; continue; }
        const int fast = (int)(e & 15u) - (d > 0.0f ? 0 : 1);
        if (fast != code) ++wrong;
        for (int j = 0; j < 15; ++j)
            if (fabs((double)q - (double)t[j]) <= 0x1p-21) ++near;
    }
    printf("%lld %lld %lld %lld %lld\n", n, wrong, near, slow, badidx);
    return 0;
}
"""


def kernel_constants():
    text = open(QUANT_CU).read()
    m = re.search(r"constexpr float kCellMagic = ([0-9.]+)f;", text)
    assert m, "kCellMagic not found in nf4_quant.cu"
    magic = float(m.group(1))
    assert magic == 16 + 1.5 * 2 ** 23
    m = re.search(r"constexpr float kGuard = (0x1p-[0-9]+)f;", text)
    assert m, "kGuard not found in nf4_quant.cu"
    guard = float.fromhex(m.group(1))
    m = re.search(r"c_cell\[64\] = \{(.*?)\};", text, flags=re.S)
    assert m, "c_cell not found in nf4_quant.cu"
    body = re.sub(r"//[^\n]*", "", m.group(1))
    cells = [int(v, 16) for v in re.findall(r"0x([0-9a-fA-F]{8})u", body)]
    assert len(cells) == 64
    return magic, guard, cells


def thresholds():
    cb = [float(v) for v in open(CODEBOOK).read().split("\n") if v.strip() and not v.startswith("#")]
    c = np.array(cb, dtype=np.float32).astype(np.float64)
    mid = (c[:-1] + c[1:]) / 2
    t = mid.astype(np.float32)
    t = np.where(t.astype(np.float64) > mid, np.nextafter(t, np.float32(-2)), t).astype(np.float32)
    assert (t.astype(np.float64) <= mid).all()
    return [float(v) for v in t]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_cell_table_code_is_exact_for_every_fp32_quotient(tmp_path):
    src = tmp_path / "cell_check.c"
    src.write_text(CHECKER)
    exe = tmp_path / "cell_check"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", str(src),
                    "-o", str(exe), "-lm"], check=True)
    magic, guard, cells = kernel_constants()
    args = [repr(magic), repr(guard)] + [hex(c) for c in cells] + [repr(v) for v in thresholds()]
    out = subprocess.run([str(exe), *args], check=True, capture_output=True, text=True, timeout=600).stdout
    n, wrong, near, slow, badidx = (int(v) for v in out.split())
    assert n == 2 * (0x3F800008 + 1)
    assert badidx == 0, f"{badidx} quotients index past cell 32"
    assert wrong == 0, f"{wrong} quotients where the fast path gives the wrong code"
    assert near == 0, f"{near} fast-path quotients within 2^-21 of a threshold"
    assert slow < n // 1000, f"{slow} quotients take the exact path"


def test_cell_entries_carry_their_threshold():
    """Each entry is a threshold T_k of the codebook, within 16 ulp, with k + 1
    in its low four bits -- and the entries step through the thresholds in
    order as the cells do."""
    _, _, cells = kernel_constants()
    t = np.array(thresholds(), dtype=np.float32)
    ks = []
    for e in cells[:33]:
        k = (e & 15) - 1
        assert 0 <= k < 15
        tb = int(t[k].view(np.uint32))
        assert abs(e - tb) < 16
        ks.append(k)
    assert ks == sorted(ks) and ks[0] == 0 and ks[-1] == 14
    assert all(c == cells[32] for c in cells[33:])


def test_cell_threshold_is_the_only_one_near_its_cell():
    """Cell c covers q in [(c - 16.5) / 16, (c - 15.5) / 16]; its entry's
    threshold T_k is the only threshold within 0.014 of that range, and
    T_(k-1) < q < T_(k+1) on it -- the two facts the code rule rests on."""
    _, _, cells = kernel_constants()
    t = np.array(thresholds(), dtype=np.float64)
    for c in range(33):
        k = (cells[c] & 15) - 1
        lo, hi = max(-1.0, (c - 16.5) / 16), min(1.0, (c - 15.5) / 16)
        assert k == 0 or t[k - 1] < lo
        assert k == 14 or t[k + 1] > hi
        for j in range(15):
            if j != k:
                assert not (lo - 0.014 <= t[j] <= hi + 0.014), (c, j)

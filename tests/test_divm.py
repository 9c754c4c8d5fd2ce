"""The group scale divides a range x = RN(max - min) of two fp16 values by
M = 2^b - 1.  The kernels compute that quotient as RN(x zh + RN(x zl)) with the
constants of kivi_divm.h (Brisebarre, Muller and Raina's division by a divisor
known in advance) instead of an IEEE division.  This test compiles the same
header on the host and checks the identity against the host's IEEE fp32
division for every fp32 x in [2^-24, 2^17] -- a superset of the ranges two fp16
values can have (0 maps to 0) -- and that the constants are the correctly
rounded zh = RN(1/M), zl = RN(1/M - zh)."""
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

from conftest import ROOT

CSRC = os.path.join(ROOT, "kivi_bit_kv_gb300", "csrc")

CHECK = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include "kivi_divm.h"
template <int B>
static unsigned long long check()
{
    unsigned long long bad = 0;
    for (uint32_t u = 0x33800000u; u <= 0x48000000u; ++u) {  // 2^-24 .. 2^17
        float x;
        memcpy(&x, &u, 4);
        volatile float p = x * kivi::DivM<B>::lo;
        const float q = fmaf(x, kivi::DivM<B>::hi, p);
        volatile float e = x / kivi::DivM<B>::M;
        bad += q != e;
    }
    return bad;
}
int main()
{
    printf("%llu %llu %llu\n", check<2>(), check<4>(), check<8>());
    printf("%a %a %a %a %a %a\n", (double)kivi::DivM<2>::hi, (double)kivi::DivM<2>::lo,
           (double)kivi::DivM<4>::hi, (double)kivi::DivM<4>::lo, (double)kivi::DivM<8>::hi,
           (double)kivi::DivM<8>::lo);
    return 0;
}
"""


def _rn_f32(q: Fraction) -> Fraction:
    """Nearest fp32 to the rational q (ties to even), by exact comparison."""
    x = np.float32(float(q))
    cands = [np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))]
    def key(c):
        return (abs(Fraction(float(c)) - q), int(np.float32(c).view(np.uint32)) & 1)
    return Fraction(float(min(cands, key=key)))


@pytest.fixture(scope="module")
def divm_output(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("divm")
    src, exe = d / "check.cc", d / "check"
    src.write_text(CHECK)
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", f"-I{CSRC}", str(src), "-o", str(exe), "-lm"],
                   check=True)
    return subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")


def test_division_by_code_range_is_correctly_rounded(divm_output):
    assert divm_output[0].split() == ["0", "0", "0"]


def test_constants_are_rounded_reciprocal_pairs(divm_output):
    vals = [Fraction(float.fromhex(v)) for v in divm_output[1].split()]
    for i, M in enumerate((3, 15, 255)):
        zh, zl = vals[2 * i], vals[2 * i + 1]
        assert zh == _rn_f32(Fraction(1, M))
        assert zl == _rn_f32(Fraction(1, M) - zh)

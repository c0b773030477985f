"""The float32 form of the normalisation product used by the CQ prepare,
row gather and Hadamard MLP kernels (needle.js "part 2", sections 1-2:
1/sqrt(n) in float64, the product taken in float64 and stored as float32).

The kernels avoid float64 arithmetic: with s = RN64(1/sqrt n) split exactly
into three float32 terms s1 + s2 + s3, they form p = RN32(v s1), its exact
error e = v s1 - p, t = RN32(RN32(v s2 + e) + v s3) and RN32(p + t).  This
test replays those steps on the host with exact intermediate arithmetic
(float64 / long double where each step's exact value fits) for every
float32 mantissa, both signs, at the binades that bound the kernels' range
for this form ([2^-60, 2^100], and signed zeros), and checks the result
against the definition RN32(RN64(v * s)).  s = RN64(1/sqrt 2) covers every odd power of
two n (the other values differ by a power of two); for even powers s is a
power of two and the product is exact.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.skipif(np.finfo(np.longdouble).nmant < 63,
                                reason="needs an 80-bit long double for the exact replay")


def split(s):
    s1 = np.float32(s)
    r = s - np.float64(s1)
    s2 = np.float32(r)
    s3 = np.float32(r - np.float64(s2))
    assert np.float64(s1) + np.float64(s2) + np.float64(s3) == s
    return s1, s2, s3


def replay(v, s1, s2, s3):
    """The kernel's steps on float32 v, each rounded exactly as the GPU does."""
    p = v * s1                                                     # RN32
    e64 = v.astype(np.float64) * np.float64(s1) - p.astype(np.float64)
    e = e64.astype(np.float32)
    assert np.array_equal(e.astype(np.float64), e64)               # the error is exact
    t1x = v.astype(np.longdouble) * np.longdouble(s2) + e.astype(np.longdouble)
    t1 = t1x.astype(np.float32)                                    # one FMA, one rounding
    t2x = v.astype(np.longdouble) * np.longdouble(s3) + t1.astype(np.longdouble)
    t2 = t2x.astype(np.float32)
    r = (p.astype(np.float64) + t2.astype(np.float64)).astype(np.float32)
    return np.copysign(r, p)  # (the kernels keep the sign of a zero product)


@pytest.mark.parametrize("k", [0, 3, 14])        # n = 2, 2^7, 2^29
@pytest.mark.parametrize("binade", [0, -60, 99])
def test_three_term_product_matches_float64_rounding(k, binade):
    s = 1.0 / np.sqrt(np.float64(2.0)) / np.float64(2.0 ** k)   # RN64(1/sqrt(2^(2k+1)))
    assert s == 1.0 / np.sqrt(np.float64(2.0 ** (2 * k + 1)))
    s1, s2, s3 = split(s)
    m = np.arange(1 << 23, dtype=np.uint32)
    for sign in (1, -1):
        v = ((np.uint32(127 + binade) << 23) | m).view(np.float32)
        if sign < 0:
            v = -v
        want = (v.astype(np.float64) * s).astype(np.float32)
        got = replay(v, s1, s2, s3)
        bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
        assert bad.size == 0, (k, binade, sign, v[bad[:3]], got[bad[:3]], want[bad[:3]])


def test_signed_zeros_keep_their_sign():
    s = 1.0 / np.sqrt(np.float64(2.0))
    s1, s2, s3 = split(s)
    v = np.array([0.0, -0.0], np.float32)
    got = replay(v, s1, s2, s3)
    assert np.array_equal(got.view(np.uint32), (v.astype(np.float64) * s).astype(np.float32).view(np.uint32))


def test_powers_of_two_are_exact():
    s = 1.0 / np.sqrt(np.float64(64.0))
    s1, s2, s3 = split(s)
    assert s1 == np.float32(0.125) and s2 == 0 and s3 == 0


def test_host_split_of_every_power_of_two(tmp_path):
    """The library's host code (make_scale) splits s = RN64(1/sqrt n) for
    every power of two n up to 2^30: the split is exact, the float32 form is
    enabled, and for odd powers the three terms are those of n = 2 scaled by
    a power of two, so the replay above covers every group and dimension."""
    import os
    import shutil
    import subprocess
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "split.cu"
    src.write_text(
        '#include <cstdio>\n#include "fwht_device.cuh"\n'
        "int main() {\n"
        "  for (int b = 0; b <= 30; b++) {\n"
        "    qmv::Scale k = qmv::make_scale(1.0 / sqrt(double(1LL << b)));\n"
        '    printf("%d %d %a %a %a %a\\n", b, k.fast, k.s, (double)k.s1, (double)k.s2, (double)k.s3);\n'
        "  }\n}\n")
    exe = tmp_path / "split"
    subprocess.run([nvcc, "-std=c++17", "-I", os.path.join(root, "quantized_weight_matvec_gb300", "csrc"),
                    "-o", str(exe), str(src)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    base = split(1.0 / np.sqrt(np.float64(2.0)))
    for line in filter(None, out):
        b, fast, s, s1, s2, s3 = line.split()
        b = int(b)
        s, s1, s2, s3 = (float.fromhex(t) for t in (s, s1, s2, s3))
        assert int(fast) == 1, b
        assert s == 1.0 / np.sqrt(np.float64(2.0 ** b))
        assert s1 + s2 + s3 == s and np.float32(s1) == s1 and np.float32(s2) == s2 and np.float32(s3) == s3
        if b % 2:
            f = 2.0 ** -(b // 2)
            assert (s1, s2, s3) == (float(base[0]) * f, float(base[1]) * f, float(base[2]) * f), b
        else:
            assert s1 == 2.0 ** -(b // 2) and s2 == 0 and s3 == 0, b

"""The kernels' division by launch-fixed divisors (csrc/fastdiv.h) against '/'.

The header has no CUDA dependency on the host side; this test compiles it
with the system C++ compiler into a small checker that compares fd_div and
fd_divmod with the hardware division over every divisor up to 4096, divisors
near powers of two up to 2^31, and dividends at both ends of [0, 2^31) plus a
seeded random sample.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "broadcast_implicit_gemm_gb300", "csrc")

CHECKER = r"""
#include <cstdio>
#include <cstdint>
#include <vector>
#include "fastdiv.h"
using namespace bigemm;
static uint64_t state = 0x9E3779B97F4A7C15ull;
static uint32_t rnd() {   // splitmix64
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return (uint32_t)((z ^ (z >> 31)) & 0x7FFFFFFFu);
}
int main() {
    std::vector<uint32_t> ds;
    for (uint32_t d = 1; d <= 4096; ++d) ds.push_back(d);
    for (int b = 12; b < 31; ++b)
        for (int k = -3; k <= 3; ++k) ds.push_back((uint32_t)((1ull << b) + k));
    ds.push_back(0x7FFFFFFFu);
    for (int i = 0; i < 2000; ++i) ds.push_back(rnd() | 1u);
    long long checked = 0;
    for (uint32_t d : ds) {
        const FastDiv f = make_fastdiv(d);
        std::vector<uint32_t> ns;
        for (uint32_t n = 0; n < 3 * d + 3 && n < 20000; ++n) ns.push_back(n);
        for (uint32_t k = 0; k < 64; ++k) ns.push_back(0x7FFFFFFFu - k);
        for (uint32_t k = 1; k < 64 && (uint64_t)k * d < 0x80000000ull; ++k) {
            ns.push_back(k * d - 1); ns.push_back(k * d);
        }
        for (int i = 0; i < 300; ++i) ns.push_back(rnd());
        for (uint32_t n : ns) {
            uint32_t r;
            const uint32_t q = fd_divmod(n, f, &r);
            if (q != n / d || r != n % d || fd_div(n, f) != n / d) {
                printf("MISMATCH n=%u d=%u q=%u r=%u\n", n, d, q, r);
                return 1;
            }
            ++checked;
        }
    }
    printf("OK %lld\n", checked);
    return 0;
}
"""


def test_fastdiv_matches_hardware_division():
    cxx = shutil.which("g++") or shutil.which("c++") or shutil.which("clang++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "chk.cc")
        exe = os.path.join(d, "chk")
        with open(src, "w") as f:
            f.write(CHECKER)
        subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert out.returncode == 0, out.stdout + out.stderr
        assert out.stdout.startswith("OK")

"""The library's division by a run-time constant (csrc/fastdiv.h), compiled
for the host with g++, against ordinary integer division: edge divisors,
the frustum strides of the workloads, and random divisors and numerators
below 2^31."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <cstdio>
#include <random>
#include "fastdiv.h"
int main() {
    std::mt19937_64 g(7);
    long bad = 0;
    const uint32_t fixed[] = {1u, 2u, 3u, 7u, 704u, 2816u, 332288u, 16384u, 45000u, 1993728u / 6u,
                              (1u << 30) + 7u, 2147483647u, 118u * 32u * 88u, 32u * 88u, 59u * 16u * 44u};
    for (uint32_t d : fixed) {
        bevpool::FastDiv f(d);
        for (uint32_t n = 0; n < 5000; ++n) bad += f.div(n) != n / d;
        for (uint32_t n = 0x7fffffffu - 5000u; n <= 0x7fffffffu - 1u; ++n) bad += f.div(n) != n / d;
        for (int i = 0; i < 200000; ++i) { uint32_t n = uint32_t(g() & 0x7fffffffu); bad += f.div(n) != n / d; }
    }
    for (int k = 0; k < 5000; ++k) {
        uint32_t d = 1u + uint32_t(g() % 0x7fffffffu);
        bevpool::FastDiv f(d);
        for (int i = 0; i < 200; ++i) { uint32_t n = uint32_t(g() & 0x7fffffffu); bad += f.div(n) != n / d; }
    }
    std::printf("%ld\n", bad);
    return bad != 0;
}
"""


def test_fastdiv_matches_integer_division(tmp_path):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    src = tmp_path / "fastdiv_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "fastdiv_check"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", os.path.join(ROOT, "depth_weighted_scatter_gb300", "csrc"),
                    str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "0", r.stdout

"""Host side of the dequantize kernels' index split: make_divu32 (csrc/mx_internal.h) builds the
multiplier and shifts of the division by an invariant integer (Granlund and Montgomery, "Division by
invariant integers using multiplication", PLDI 1994, section 4) that every 32-bit dequantize thread
uses to find its row and group.  A small host program compiled against the header checks
q = (t + ((n - t) >> s1)) >> s2, t = mulhi(m, n), against exact integer division for the divisors the
library passes (row widths in blocks, group and scale row counts), powers of two and their neighbours,
and random 32-bit divisors, each with the edge and random numerators.  No GPU is needed."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "microscaled_precision_numerics_gb300", "csrc")

PROGRAM = r"""
#include "mx_internal.h"
#include <cstdio>
#include <cstdint>

static uint32_t div_host(uint32_t n, mxk::DivU32 d) {
    const uint32_t t = (uint32_t)(((uint64_t)n * d.m) >> 32);
    return (t + ((n - t) >> d.s1)) >> d.s2;
}

int main() {
    uint64_t state = 0x9E3779B97F4A7C15ull;
    auto next = [&]() { state ^= state << 13; state ^= state >> 7; state ^= state << 17; return state; };
    uint64_t divisors[400];
    int nd = 0;
    const uint64_t fixed[] = {1, 2, 3, 5, 7, 48, 64, 96, 128, 129, 256, 768, 1536, 2048, 2064, 4096, 8192, 12288,
                              14336, 65535, 65536, 65537, 0x7FFFFFFFull, 0x80000000ull, 0x80000001ull, 0xFFFFFFFFull};
    for (uint64_t d : fixed) divisors[nd++] = d;
    for (int k = 1; k < 32; ++k) {
        divisors[nd++] = (1ull << k) - 1;
        divisors[nd++] = (1ull << k) + 1;
    }
    while (nd < 400) divisors[nd++] = 1 + next() % 0xFFFFFFFFull;
    long checked = 0;
    for (int i = 0; i < nd; ++i) {
        const uint64_t d = divisors[i];
        const mxk::DivU32 dv = mxk::make_divu32(d);
        uint64_t ns[32] = {0, 1, d - 1, d, d + 1, 2 * d - 1, 2 * d, 0xFFFFFFFFull, 0xFFFFFFFEull, 0x80000000ull,
                           0x7FFFFFFFull};
        for (int j = 11; j < 32; ++j) ns[j] = next() & 0xFFFFFFFFull;
        for (int j = 0; j < 32; ++j) {
            if (ns[j] > 0xFFFFFFFFull) continue;
            const uint32_t n = (uint32_t)ns[j];
            if (div_host(n, dv) != (uint32_t)(n / d)) {
                std::printf("mismatch n=%u d=%llu\n", n, (unsigned long long)d);
                return 1;
            }
            ++checked;
        }
        for (uint32_t n = 0; n < 4096; ++n) {
            if (div_host(n, dv) != (uint32_t)(n / d)) {
                std::printf("mismatch n=%u d=%llu\n", n, (unsigned long long)d);
                return 1;
            }
            ++checked;
        }
    }
    std::printf("ok %ld\n", checked);
    return 0;
}
"""


def test_make_divu32_matches_integer_division():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "divisor_check.cu")
        exe = os.path.join(tmp, "divisor_check")
        with open(src, "w") as f:
            f.write(PROGRAM)
        # the header's device helpers use sm_103a instructions; the program itself runs on the host only
        build = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O2",
                                "-I", CSRC, "-I", os.path.join(ROOT, "include"), src, "-o", exe],
                               capture_output=True, text=True, timeout=300)
        assert build.returncode == 0, build.stderr[-2000:]
        run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert run.returncode == 0 and run.stdout.startswith("ok"), run.stdout + run.stderr

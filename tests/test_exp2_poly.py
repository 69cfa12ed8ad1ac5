"""The FMA-pipe exp2 of csrc/exp2_poly.h, on the host (no GPU).

The kernel's packed version rounds lane by lane exactly as the scalar function
does (add.rn / fma.rn per lane), so evaluating the scalar function compiled for
the host checks the arithmetic the GPU performs.  Against the C library's
exp2 in double precision, over every seventh fp32 bit pattern of [-126, 64.5]
(the exponents the softmax can produce: the stale-maximum threshold keeps
them at most its T <= 64, and anything below -126 underflows):
  - the relative error stays within the fp32 evaluation of the minimax fit;
  - integers n give exactly 2^n, and 0 gives exactly 1;
  - -inf, -127 and everything below give exactly +0 (masked scores);
  - (-127, -126) gives a value in [0, 2^-125].
"""
import json
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "exact_long_sequence_gb300", "csrc")

# Largest relative error of the fp32 evaluation (fit_exp2_poly.py prints the same
# figures on [-1/2, 1/2]), with a little room for the range reduction's rounding.
BOUND = {3: 1.02e-4, 4: 2.95e-6, 5: 1.7e-7}

PROGRAM = r"""
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include "exp2_poly.h"

static float from_bits(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
static uint32_t to_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }

int main() {
    using elsattn::exp2_poly;
    double worst = 0.0, worst_x = 0.0;
    long count = 0;
    // negative x in [-126, -0]: bit patterns 0x80000000 .. bits(-126)
    const uint32_t neg_end = to_bits(-126.0f);
    for (uint64_t u = 0x80000000u; u <= neg_end; u += 7) {
        const float x = from_bits((uint32_t)u);
        const double e = std::fabs((double)exp2_poly(x) / std::exp2((double)x) - 1.0);
        if (e > worst) { worst = e; worst_x = x; }
        ++count;
    }
    const uint32_t pos_end = to_bits(64.5f);
    for (uint64_t u = 0; u <= pos_end; u += 7) {
        const float x = from_bits((uint32_t)u);
        const double e = std::fabs((double)exp2_poly(x) / std::exp2((double)x) - 1.0);
        if (e > worst) { worst = e; worst_x = x; }
        ++count;
    }
    int integers_exact = 1;
    for (int n = -126; n <= 8; ++n)
        if (exp2_poly((float)n) != std::ldexp(1.0f, n)) integers_exact = 0;
    const float zeros_in[] = {-INFINITY, -1e30f, -4194304.0f, -1000.0f, -200.0f, -127.5f, -127.0f};
    int zeros_exact = 1;
    for (float z : zeros_in)
        if (to_bits(exp2_poly(z)) != 0u) zeros_exact = 0;
    int gap_ok = 1;
    for (float x = -126.999f; x < -126.0f; x += 0.001f) {
        const float y = exp2_poly(x);
        if (!(y >= 0.0f && y <= std::ldexp(1.0f, -125))) gap_ok = 0;
    }
    std::printf("{\"worst\": %.6e, \"worst_x\": %.9g, \"count\": %ld, \"one\": %d, \"integers_exact\": %d, "
                "\"zeros_exact\": %d, \"gap_ok\": %d}\n",
                worst, worst_x, count, exp2_poly(0.0f) == 1.0f, integers_exact, zeros_exact, gap_ok);
    return 0;
}
"""


@pytest.fixture(scope="module")
def build_dir(tmp_path_factory):
    d = tmp_path_factory.mktemp("exp2poly")
    (d / "probe.cpp").write_text(PROGRAM)
    return d


@pytest.mark.parametrize("degree", [3, 4, 5])
def test_exp2_poly_against_libm(build_dir, degree):
    exe = build_dir / f"probe{degree}"
    subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", f"-DELS_EXP2_POLY_DEGREE={degree}",
                    "-I", HEADER_DIR, str(build_dir / "probe.cpp"), "-o", str(exe)], check=True)
    r = json.loads(subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout)
    print(f"degree {degree}: {r}")
    assert r["count"] > 100_000_000
    assert r["worst"] <= BOUND[degree], r
    assert r["one"] == 1 and r["integers_exact"] == 1 and r["zeros_exact"] == 1 and r["gap_ok"] == 1, r

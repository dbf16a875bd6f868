"""The multiply-shift divider used for row indexing (sms_fastdiv.h) against
exact integer division, compiled as plain host C++ (no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "scaled_masked_softmax_gb300", "csrc")

CHECK = r"""
#include "sms_fastdiv.h"
#include <cstdio>
#include <cstdint>
int main() {
    uint64_t bad = 0, n_checked = 0;
    uint64_t s = 88172645463325252ull;  // xorshift64 state
    auto rnd = [&]() { s ^= s << 13; s ^= s >> 7; s ^= s << 17; return s; };
    const uint32_t ds[] = {1u, 2u, 3u, 5u, 7u, 64u, 100u, 127u, 128u, 1000u, 1023u, 1024u, 1025u, 2048u, 4096u,
                           4099u, 8192u, 16384u, 65535u, 65536u, 1u << 20, (1u << 30) - 1, 1u << 30,
                           (1u << 31) - 1, 1u << 31};
    for (uint32_t d : ds) {
        sms::FastDiv f(d);
        const uint32_t edge[] = {0u, 1u, d - 1, d, d + 1, 2 * d - 1, 2 * d, 0xffffffffu, 0xfffffffeu,
                                 0x7fffffffu, 0x80000000u};
        for (uint32_t n : edge) { ++n_checked; if (f.div(n) != n / d) ++bad; }
        for (int i = 0; i < 200000; ++i) {
            uint32_t n = (uint32_t)rnd();
            ++n_checked;
            if (f.div(n) != n / d) ++bad;
        }
    }
    for (int i = 0; i < 2000000; ++i) {
        uint32_t d = (uint32_t)(rnd() >> (33 + rnd() % 31));
        if (!d) d = 1;
        uint32_t n = (uint32_t)rnd();
        sms::FastDiv f(d);
        ++n_checked;
        if (f.div(n) != n / d) ++bad;
    }
    std::printf("%llu %llu\n", (unsigned long long)n_checked, (unsigned long long)bad);
    return bad != 0;
}
"""


def test_fastdiv_matches_exact_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "check.cpp"
    src.write_text(CHECK)
    exe = tmp_path / "check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    n, bad = map(int, out.stdout.split())
    assert n > 5_000_000 and bad == 0, out.stdout

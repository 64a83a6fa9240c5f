"""The decode kernel's static page partition (partition.cuh), compiled for the
host with g++ and checked exhaustively: every CTA gets a non-empty contiguous
range of P/C pages (+-1), the ranges tile [0, P) in order, and cta_of inverts
them."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_kv_cache_fp8kv_gb300", "csrc")

CHECKER = r"""
#include <cstdio>
#include <cstdlib>
#include "partition.cuh"
using namespace fp8kv;
static int check(long long P, int C) {
    const Partition q = make_partition(P, C);
    if (range_start(q, 0) != 0 || range_start(q, C) != P) return 1;
    long long prev = 0;
    for (int c = 0; c < C; ++c) {
        const long long a = range_start(q, c), b = range_start(q, c + 1);
        if (b <= a || a != prev) return 2;            // non-empty, contiguous, in order
        prev = b;
        // cta_of at both ends and the middle of the range
        const long long ps[3] = {a, b - 1, a + (b - a) / 2};
        for (long long p : ps) if (cta_of(q, p) != c) return 3;
    }
    if (P <= 20000)
        for (long long p = 0, c = 0; p < P; ++p) {
            while (range_start(q, c + 1) <= p) ++c;
            if (cta_of(q, p) != c) return 4;
        }
    for (int c = 0; c < C; ++c) {
        const long long n = range_start(q, c + 1) - range_start(q, c);
        if (n < P / C || n > P / C + 1) return 5;     // equal shares
    }
    return 0;
}
int main() {
    long long Ps[] = {1, 2, 3, 7, 16, 63, 64, 100, 304, 305, 607, 608, 1000, 4096, 19455, 19456, 19457,
                      65536, 83114, 1000003, 10000019, (1ll << 33) + 17};
    int Cs[] = {1, 2, 3, 5, 16, 151, 152, 303, 304, 512, 1024};
    int fails = 0;
    for (long long P : Ps)
        for (int C : Cs) {
            if (C > P) continue;
            const int r = check(P, C);
            if (r) { printf("FAIL P=%lld C=%d code=%d\n", P, C, r); ++fails; }
        }
    printf("%s\n", fails ? "FAILED" : "OK");
    return fails != 0;
}
"""


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    d = tmp_path_factory.mktemp("partition")
    src = d / "check.cpp"
    src.write_text(CHECKER)
    exe = d / "check"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return exe


def test_partition_ranges_tile_the_pages_and_invert(checker):
    r = subprocess.run([str(checker)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout
    assert r.stdout.strip().endswith("OK")

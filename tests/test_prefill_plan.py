"""The prefill's key-range split plan (prefill_plan.h), compiled for the host
with g++: no split once the units fill a wave of resident CTAs, the limits
(at most 64 splits, at least 8 pages each), one full wave when the pages are
plentiful, and no choice whose wave count the model would beat by splitting
less."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_kv_cache_fp8kv_gb300", "csrc")

CHECKER = r"""
#include <cstdio>
#include "prefill_plan.h"
using namespace fp8kv::prefill;
int main() {
    int fails = 0;
    const long long units_list[] = {1, 2, 7, 8, 16, 63, 64, 100, 255, 256, 303, 304, 305, 1000, 4096};
    const long long pages_list[] = {1, 7, 8, 15, 16, 100, 313, 1375, 8192, 100000};
    const long long slots_list[] = {152, 304, 456, 608};
    for (long long slots : slots_list)
        for (long long units : units_list)
            for (long long pages : pages_list) {
                const int s = choose_splits(units, pages, slots);
                if (s < 1 || s > kMaxSplits) { printf("FAIL range u=%lld p=%lld s=%lld -> %d\n", units, pages, slots, s); ++fails; }
                if (s > 1 && (long long)s * kMinSplitPages > pages) { printf("FAIL min pages u=%lld p=%lld -> %d\n", units, pages, s); ++fails; }
                if (units >= slots && s != 1) { printf("FAIL full wave u=%lld slots=%lld -> %d\n", units, slots, s); ++fails; }
            }
    // one unit per kv head of a single long sequence: one full wave of splits
    if (choose_splits(8, 8192, 304) != 38) { printf("FAIL 8 units x 8192 pages -> %d\n", choose_splits(8, 8192, 304)); ++fails; }
    if (choose_splits(4, 100000, 152) != 38) { printf("FAIL 4 units -> %d\n", choose_splits(4, 100000, 152)); ++fails; }
    // a single unit with few pages: bounded by the minimum split size
    if (choose_splits(1, 100, 304) != 12) { printf("FAIL 1 unit x 100 pages -> %d\n", choose_splits(1, 100, 304)); ++fails; }
    // too few pages to split
    if (choose_splits(1, 15, 304) != 1) { printf("FAIL 15 pages -> %d\n", choose_splits(1, 15, 304)); ++fails; }
    printf("%s\n", fails ? "FAILED" : "OK");
    return fails != 0;
}
"""


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    d = tmp_path_factory.mktemp("prefill_plan")
    src = d / "check.cpp"
    src.write_text(CHECKER)
    exe = d / "check"
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], capture_output=True,
                       text=True)
    if r.returncode != 0:
        pytest.fail("g++ failed:\n" + r.stderr)
    return str(exe)


def test_split_plan_properties(checker):
    r = subprocess.run([checker], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout[-2000:]

"""The decode kernel's walk over a CTA's page range and its per-warp windows
(walk.cuh), compiled for the host with g++ and checked on many random and
edge-case lengths:

* the segments of all CTAs tile every unit's pages exactly once, in order;
* each segment's warp shares tile the segment, the last warp's share holding
  the segment's last page;
* the issue side (windows of <= 32 pages, cut into stages of PPS pages) visits
  exactly the compute side's stages, in the same order, for every warp;
* the page that receives a decode step's new rows (each unit's last page) is
  flagged in exactly one window, at its last position.
"""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_kv_cache_fp8kv_gb300", "csrc")

CHECKER = r"""
#include <cstdio>
#include <cstdlib>
#include <vector>
#include <random>
#include "partition.cuh"
#include "walk.cuh"
using namespace fp8kv;

struct Page { int b, hk; int64_t idx; };   // page idx (0-based) of unit (b, hk)

static int check(const std::vector<int>& n_b, int Hkv, int C, int NW, int PPS) {
    const int B = (int)n_b.size();
    std::vector<int32_t> pre(B + 1, 0);
    for (int b = 0; b < B; ++b) pre[b + 1] = pre[b] + n_b[b];
    const int64_t P = (int64_t)Hkv * pre[B];
    if (P == 0) return 0;
    const int Ce = (int)(P < C ? P : C);
    const Partition part = make_partition(P, Ce);
    std::vector<std::vector<int>> seen(B * Hkv);
    std::vector<int> last_flags(B * Hkv, 0);
    for (int b = 0; b < B; ++b) for (int h = 0; h < Hkv; ++h) seen[b * Hkv + h].assign(n_b[b], 0);
    for (int c = 0; c < Ce; ++c) {
        const int64_t s = range_start(part, c), e = range_start(part, c + 1);
        // compute side: segments in order
        std::vector<std::vector<std::vector<Page>>> comp(NW);   // per warp: stages
        Walker w;
        walk_start(w, pre.data(), B, Hkv, s);
        int64_t covered = 0;
        while (true) {
            const int np = seg_pages(w, e);
            if (np <= 0) return 10;
            if (w.g < w.base || w.g + np > w.base + w.n) return 11;
            int prev_hi = 0;
            for (int wp = 0; wp < NW; ++wp) {
                int q0, q1;
                warp_share(w, e, wp, NW, q0, q1);
                if (q0 != prev_hi || q1 < q0) return 12;
                prev_hi = q1;
                for (int p0 = q0; p0 < q1; p0 += PPS) {
                    std::vector<Page> st;
                    for (int p = p0; p < q1 && p < p0 + PPS; ++p) st.push_back({w.b, w.hk, w.g - w.base + p});
                    comp[wp].push_back(st);
                }
                if (wp == NW - 1 && q1 != np) return 13;
            }
            for (int p = 0; p < np; ++p) {
                int& x = seen[w.b * Hkv + w.hk][w.g - w.base + p];
                if (x) return 14;
                x = 1;
            }
            covered += np;
            if (seg_is_last(w, e)) break;
            walk_next(w, pre.data(), Hkv);
        }
        if (covered != e - s) return 15;
        // issue side: windows
        for (int wp = 0; wp < NW; ++wp) {
            Walker w0;
            walk_start(w0, pre.data(), B, Hkv, s);
            WinPos cur = first_window_from(w0, true, pre.data(), Hkv, e, wp, NW);
            size_t k = 0;
            while (cur.valid) {
                if (cur.n < 1 || cur.n > 32 || cur.start + cur.n > cur.hi) return 20;
                const bool last = window_holds_unit_end(cur, e);
                if (last) last_flags[cur.w.b * Hkv + cur.w.hk]++;
                for (int cpos = 0; cpos < cur.n; cpos += PPS) {
                    const int n = cur.n - cpos < PPS ? cur.n - cpos : PPS;
                    if (k >= comp[wp].size()) return 21;
                    const std::vector<Page>& st = comp[wp][k++];
                    if ((int)st.size() != n) return 22;
                    for (int p = 0; p < n; ++p) {
                        const Page& q = st[p];
                        const int64_t idx = cur.w.g - cur.w.base + cur.start + cpos + p;
                        if (q.b != cur.w.b || q.hk != cur.w.hk || q.idx != idx) return 23;
                        const bool is_unit_last = idx == cur.w.n - 1;
                        const bool flagged = last && cur.start + cpos + p == cur.hi - 1;
                        if (is_unit_last != flagged) return 24;
                    }
                }
                cur = next_window(cur, pre.data(), Hkv, e, wp, NW);
            }
            if (k != comp[wp].size()) return 25;
        }
    }
    for (int u = 0; u < B * Hkv; ++u) {
        for (int x : seen[u]) if (!x) return 30;
        if (!seen[u].empty() && last_flags[u] != 1) return 31;
        if (seen[u].empty() && last_flags[u] != 0) return 32;
    }
    return 0;
}

int main() {
    std::mt19937_64 rng(7);
    int fails = 0, cases = 0;
    const int Cs[] = {1, 2, 3, 7, 64, 151, 152, 303, 304, 1024};
    const int NWs[] = {1, 2, 3, 4, 6, 8};
    const int PPSs[] = {1, 2, 4};
    for (int it = 0; it < 160; ++it) {
        const int B = 1 + (int)(rng() % 12);
        const int Hkv = 1 << (rng() % 4);
        std::vector<int> n_b(B);
        const int kind = it % 4;
        for (int b = 0; b < B; ++b) {
            if (kind == 0) n_b[b] = (int)(rng() % 5);                 // tiny, some empty
            else if (kind == 1) n_b[b] = (int)(rng() % 70);
            else if (kind == 2) n_b[b] = 1000 + (int)(rng() % 400);    // ~20K tokens
            else n_b[b] = (rng() % 3 == 0) ? 0 : (int)(rng() % 3000);
        }
        for (int C : Cs)
            for (int NW : NWs)
                for (int PPS : PPSs) {
                    ++cases;
                    const int r = check(n_b, Hkv, C, NW, PPS);
                    if (r) {
                        if (fails < 20) printf("FAIL it=%d B=%d Hkv=%d C=%d NW=%d PPS=%d code=%d\n", it, B, Hkv, C, NW, PPS, r);
                        ++fails;
                    }
                }
    }
    // one long sequence (131072 tokens, 8 heads) over a full grid
    for (int NW : NWs) for (int PPS : PPSs) {
        ++cases;
        const int r = check(std::vector<int>{8192}, 8, 304, NW, PPS);
        if (r) { printf("FAIL long NW=%d PPS=%d code=%d\n", NW, PPS, r); ++fails; }
    }
    printf("%d cases, %s\n", cases, fails ? "FAILED" : "OK");
    return fails != 0;
}
"""


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    d = tmp_path_factory.mktemp("walk")
    src = d / "check.cpp"
    src.write_text(CHECKER)
    exe = d / "check"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return exe


def test_warp_windows_match_the_compute_walk_and_tile_every_page(checker):
    r = subprocess.run([str(checker)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout
    assert r.stdout.strip().endswith("OK")

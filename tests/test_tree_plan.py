"""Host logic of the tree executor's grid (csrc/tree_plan.h), no GPU: the
header compiles as plain C++, and its closed forms are checked against the
definitions for every p <= 1024 ("Derive the cost of a ring all-reduce",
tree all-reduce: reduce up a binary tree, broadcast down):
  - rank r is a parent at reduce level l iff r mod 2^(l+1) == 0 and
    r + 2^l < p, and those levels are 0 .. m - 1;
  - w_r = m_r + (1 unless r is the root); the w_r add up to 2 (p - 1), one
    per hop of the schedule (p - 1 reduce hops, p - 1 broadcast hops);
  - the first CTA of rank r is scale * (w_0 + ... + w_(r-1)), and mapping a
    CTA index back to its rank by binary search over those starts gives each
    rank exactly scale * w_r CTAs."""
import os
import subprocess
import tempfile

from tests.conftest import ROOT

PROGRAM = r'''
#include <cstdio>
#include "tree_plan.h"
using namespace rar;
static int parent_levels(int r, int p, int L) {  // by definition
    int m = 0;
    for (int l = 0; l < L; l++)
        if (r % (1 << (l + 1)) == 0 && r + (1 << l) < p) m++;
    return m;
}
int main() {
    long long bad = 0;
    for (int p = 2; p <= 1024; p++) {
        const int L = tree_levels(p);
        if ((1 << L) < p || (L > 0 && (1 << (L - 1)) >= p)) bad++;
        long long acc = 0;
        for (int r = 0; r < p; r++) {
            const int m = tree_reduce_levels(r, p, L);
            if (m != parent_levels(r, p, L)) bad++;
            for (int l = 0; l < m; l++)  // the parent levels are 0 .. m - 1
                if (!(r % (1 << (l + 1)) == 0 && r + (1 << l) < p)) bad++;
            if (tree_weight(r, p, L) != m + (r ? 1 : 0)) bad++;
            for (int scale = 1; scale <= 3; scale++)
                if (tree_first_cta(r, p, L, scale, 0) != acc * scale) bad++;
            if (tree_first_cta(r, p, L, 0, 5) != 5LL * r) bad++;
            acc += tree_weight(r, p, L);
        }
        if (acc != 2LL * (p - 1)) bad++;
        // every CTA maps back to a rank, each rank gets scale * w_r CTAs
        const int scale = 2;
        const long long total = tree_first_cta(p, p, L, scale, 0);
        if (total != 2LL * scale * (p - 1)) bad++;
        long long owned_prev = -1;
        int count = 0, cur = 0;
        for (long long b = 0; b < total; b++) {
            int lo = 0, hi = p - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) / 2;
                if (tree_first_cta(mid, p, L, scale, 0) <= b) lo = mid;
                else hi = mid - 1;
            }
            if (lo != cur) {
                if (count != scale * tree_weight(cur, p, L)) bad++;
                if (lo != cur + 1) bad++;
                cur = lo;
                count = 0;
            }
            count++;
            (void)owned_prev;
        }
        if (cur != p - 1 || count != scale * tree_weight(p - 1, p, L)) bad++;
    }
    std::printf("%lld\n", bad);
    return bad != 0;
}
'''


def test_tree_plan_closed_forms_match_the_definitions():
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "plan.cpp")
        exe = os.path.join(d, "plan")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run(["g++", "-std=c++17", "-O2", "-I", os.path.join(ROOT, "ring_all_reduce_rar_gb300", "csrc"),
                        src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "0", out.stdout

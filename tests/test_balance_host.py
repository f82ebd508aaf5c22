"""The balanced grid's partition arithmetic (gt_tc_common.cuh: Balance,
piece_of, cta_of, share_of), compiled for the host with nvcc and checked
exhaustively over grid shapes: every (task, KV block) step is covered by
exactly one share, a share meets at most two tasks, cta_of finds the share
that holds a step, and with an even CTA count (the only kind balance_grid
makes) share_of is a permutation of the CTAs and shares k and k + ctas / 2
start at the same step of the two halves.
No GPU is needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "graph_transformer_attention_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r'''
#include <cstdio>
#include <vector>
#include "gt_tc_common.cuh"
using gt::tc::Balance;
using gt::tc::Piece;
using gt::tc::piece_of;

static int check(int tiles, int nblk, int ctas) {
    const int tasks = 2 * tiles;
    Balance bl{ctas, tasks, nblk};
    std::vector<int> owner((size_t)tasks * nblk, -1);
    std::vector<int> seen(ctas, 0);
    if (ctas % 2 == 0)                                           // the grids are even (balance_grid)
        for (int b = 0; b < ctas; ++b) {
            const int c = bl.share_of(b);
            if (c < 0 || c >= ctas || seen[c]++) return 1;      // share_of is a permutation
        }
    for (int c = 0; c < ctas; ++c) {
        int pieces = 0;
        for (int which = 0; which < 2; ++which) {   // a third task's steps would stay uncovered (6)
            Piece p;
            if (!piece_of(bl, c, which, p)) break;
            ++pieces;
            if (p.task < 0 || p.task >= tasks || p.b0 < 0 || p.b0 >= p.b1 || p.b1 > nblk) return 2;
            for (int s = p.b0; s < p.b1; ++s) {
                const long long step = (long long)p.task * nblk + s;
                if (owner[step] != -1) return 3;                 // covered once
                owner[step] = c;
                if (bl.cta_of(step) != c) return 4;              // cta_of finds the share
            }
        }
        if (pieces < 1) return 5;
    }
    for (size_t s = 0; s < owner.size(); ++s)
        if (owner[s] < 0) return 6;
    if (ctas % 2 == 0)
        for (int c = 0; c < ctas / 2; ++c)
            if (bl.lo(c) + bl.total() / 2 != bl.lo(c + ctas / 2)) return 7;
    return 0;
}

int main() {
    int cases = 0;
    const int tiles_list[] = {1, 2, 3, 5, 24, 53, 78, 128, 157, 256};
    const int nblk_list[] = {1, 2, 7, 16, 64, 155, 256, 313};
    for (int tiles : tiles_list)
        for (int nblk : nblk_list) {
            const int tasks = 2 * tiles;
            // every CTA count from one per task up to one per step (even and odd)
            for (long long g = tasks; g <= (long long)tasks * nblk && g <= 2 * tasks + 640; ++g) {
                const int rc = check(tiles, nblk, (int)g);
                if (rc) { printf("fail %d tiles=%d nblk=%d ctas=%lld\n", rc, tiles, nblk, g); return 1; }
                ++cases;
            }
        }
    printf("ok %d\n", cases);
    return 0;
}
'''


def test_balanced_partition_invariants(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "balance_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "balance_check"
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-I", INCLUDE, "-I", CSRC, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout + out.stderr

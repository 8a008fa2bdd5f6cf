"""Index arithmetic of the one-pass row kernel's work split, checked on the host.

The kernel splits U = tasks x chunks units over W warps by w U / W, finds a
unit's warp by the inverse formula, writes each (warp, row part) list to slot
w Pw + (t - first row of w), and lets the warp that completes a row's part
count merge the parts of warps split_owner(first chunk) .. split_owner(last
chunk).  These checks restate those formulas in integer arithmetic (all
operands are non-negative, so floor division matches C) and prove over many
shapes that the ranges partition the units, that the owner formula inverts the
split, that part slots are distinct and inside the workspace's
tasks + 3 x kMaxRowWarps partial lists, and that the part count a row waits
for is the number of warps that touch it.  The constants are read from the
sources.
"""
import os
import random
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_verification_rows_gb300", "csrc")


def _const(fname, name):
    text = open(os.path.join(CSRC, fname)).read()
    m = re.search(r"constexpr int " + name + r" = ([^;]+);", text)
    assert m, name
    return m.group(1)


K_FAST_VECS = int(_const("sv_internal.cuh", "kFastVecs"))
K_MAX_ROW_WARPS = int(_const("sv_internal.cuh", "kMaxRowWarps"))
assert _const("sv_fast.cu", "kWarpChunkBytes").startswith("32 * kFastVecs * 16")
CHUNK_BYTES = 32 * K_FAST_VECS * 16


def split(n_tasks, vocab, esz, max_warps):
    nc = (vocab + CHUNK_BYTES // esz - 1) // (CHUNK_BYTES // esz)
    U = n_tasks * nc
    W = min(max_warps, U)
    Pw = ((U + W - 1) // W + nc - 1) // nc + 1
    lo = lambda w: w * U // W
    owner = lambda g: ((g + 1) * W + U - 1) // U - 1
    slot = lambda w, t: w * Pw + (t - lo(w) // nc)
    return nc, U, W, Pw, lo, owner, slot


def check(n_tasks, vocab, esz, max_warps):
    nc, U, W, Pw, lo, owner, slot = split(n_tasks, vocab, esz, max_warps)
    assert lo(0) == 0 and lo(W) == U
    touching = {}
    slots = set()
    for w in range(W):
        a, b = lo(w), lo(w + 1)
        assert a < b                                   # W <= U: every warp has a unit
        assert owner(a) == w and owner(b - 1) == w     # the inverse formula
        if a > 0:
            assert owner(a - 1) == w - 1
        for t in range(a // nc, (b - 1) // nc + 1):
            s = slot(w, t)
            assert 0 <= t - a // nc < Pw               # a warp's parts stay in its own slots
            assert 0 <= s < W * Pw and s not in slots
            slots.add(s)
            touching.setdefault(t, []).append(w)
    assert W * Pw <= n_tasks + 3 * K_MAX_ROW_WARPS     # the workspace's partial lists
    for t in range(n_tasks):
        g0 = t * nc
        first, last = owner(g0), owner(g0 + nc - 1)
        assert touching[t] == list(range(first, last + 1))
        assert last - first + 1 == len(touching[t])    # the count the last part waits for


@pytest.mark.parametrize("esz", [2, 4])
def test_small_shapes_exhaustively(esz):
    for n_tasks in range(1, 24):
        for vocab in (1, 2, 7, 1023, 1024, 1025, 2047, 2048, 2049, 4096, 5000, 20_000):
            for max_warps in (1, 2, 3, 16, 17, 64, 2432, K_MAX_ROW_WARPS):
                check(n_tasks, vocab, esz, max_warps)


def test_benchmark_shapes():
    check(1920, 248_320, 2, 2432)       # 1,024 target + 896 draft rows on 152 SMs x 16 warps
    check(4096, 129_280, 2, 2432)       # greedy rows
    check(1024, 248_320, 2, 2432)


def test_random_shapes():
    rng = random.Random(7)
    for _ in range(300):
        check(rng.randint(1, 3000), rng.randint(1, 300_000), rng.choice([2, 4]),
              rng.choice([16 * rng.randint(1, 256), rng.randint(1, K_MAX_ROW_WARPS)]))

"""Split-KV planning (the decode's integer step) checked on the host.

tests/plan_check.cu compiles the planning helpers of csrc/plan.cuh for the CPU
(nvcc; no GPU involved) and prints what they return for each batch.  The
checks below restate, from the definitions, what the decode kernels need:
tiles of ceil(L / tile) tokens in batch order; the even split of the tile
list; the sequence-aligned plan w_b = min(t_b, 1 + floor((G - n) t_b / T))
(1 when G <= n); every tile processed exactly once under either plan; one
partial slot per segment, unique and inside the G + B slots of the
workspace; and the combine's slot set for each sequence (workers without
tiles skipped) equal to the slots its segments wrote.
"""
import json
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SEG_PENALTY_TILES = 3


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    out = tmp_path_factory.mktemp("plan") / "plan_check"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
                    os.path.join(ROOT, "tests", "plan_check.cu"), "-o", str(out)],
                   check=True, capture_output=True, text=True)
    return str(out)


def run_cases(harness, cases):
    lines = [str(len(cases))]
    for G, tile, L in cases:
        lines.append(" ".join(str(v) for v in [len(L), G, tile] + list(L)))
    r = subprocess.run([harness], input="\n".join(lines) + "\n", capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    out = [json.loads(x) for x in r.stdout.splitlines()]
    assert len(out) == len(cases)
    return out


def expected_entries(t, T, n, G):
    if t == 0:
        return 0
    if G <= n:
        return 1
    return min(t, 1 + (G - n) * t // T)


def simulate(res, G, B, aligned):
    """Worker ranges and partial slots as the partial kernels derive them."""
    pre, W, wb = res["pre"], res["W"], res["worker_begin"]
    E = W[B]
    eot_off = np.concatenate([[0], np.cumsum(np.diff(pre))]).astype(int)
    segs = []
    for g in range(G):
        if aligned:
            lo, hi = res["entry_tile"][g * E // G], res["entry_tile"][(g + 1) * E // G]
        else:
            lo, hi = wb[g], wb[g + 1]
        x = lo
        while x < hi:
            b = res["seq_of_tile"][x]
            e = min(pre[b + 1], hi)
            if aligned:
                slot = W[b] + res["entry_of_tile"][eot_off[b] + (x - pre[b])]
            else:
                slot = g + b
            segs.append((g, b, x, e, slot))
            x = e
    return segs


def check_case(G, tile, L, res):
    B = len(L)
    t = [(l + tile - 1) // tile for l in L]
    pre = [0] + list(np.cumsum(t))
    T, n = pre[-1], sum(1 for v in t if v > 0)
    assert res["pre"] == pre and res["T"] == T and res["n"] == n
    # ---- sequence-aligned plan
    w = [expected_entries(tb, T, n, G) for tb in t]
    W = [0] + list(np.cumsum(w))
    E = W[-1]
    assert res["W"] == W
    for tb, wb_ in zip(t, w):
        assert (tb == 0 and wb_ == 0) or 1 <= wb_ <= tb
    assert E <= max(G, n)
    starts = []
    for b in range(B):
        for k in range(w[b]):
            starts.append(pre[b] + t[b] * k // w[b])
            assert res["seq_of_entry"][W[b] + k] == b
    assert res["entry_tile"] == starts + [T]
    assert all(a < c for a, c in zip(starts, starts[1:] + [T]))        # no entry is empty
    eot = []
    for b in range(B):
        bounds = [t[b] * k // w[b] for k in range(w[b] + 1)] if w[b] else [0]
        for tau in range(t[b]):
            eot.append(next(k for k in range(w[b]) if bounds[k] <= tau < bounds[k + 1]))
    assert res["entry_of_tile"] == eot
    # ---- tile list, even split
    assert res["seq_of_tile"] == [b for b in range(B) for _ in range(t[b])]
    wbeg = [g * T // G for g in range(G + 1)]
    assert res["worker_begin"] == wbeg
    sizes = np.diff(wbeg)
    assert T == 0 or sizes.max() - sizes.min() <= 1
    assert res["worker_of"] == [max(g for g in range(G) if wbeg[g] <= x) for x in range(T)]
    # ---- the plan choice
    cost = max([-(-t[b] // w[b]) for b in range(B) if w[b]], default=0)
    assert res["cost"] == cost
    if T == 0:
        want = True
    else:
        q = -(-T // G)
        t_min = min(v for v in t if v > 0)
        want = cost <= q + SEG_PENALTY_TILES * (-(-q // t_min))
    assert res["aligned"] == int(want)
    # ---- both plans: coverage, slots, what the combine reads
    for aligned in (True, False):
        segs = simulate(res, G, B, aligned)
        covered = sorted(x for (_, _, lo, hi, _) in segs for x in range(lo, hi))
        assert covered == list(range(T)), "every tile exactly once"
        slots = [s for (*_, s) in segs]
        assert len(set(slots)) == len(slots) and all(0 <= s < G + B for s in slots)
        for b in range(B):
            written = sorted(s for (_, bb, _, _, s) in segs if bb == b)
            if t[b] == 0:
                assert written == []
                continue
            if aligned:
                read = list(range(W[b], W[b] + w[b]))
            else:
                # the owners of b's first and last tiles and every worker between
                # them that has tiles at all (an idle worker writes nothing)
                g0, g1 = res["worker_of"][pre[b]], res["worker_of"][pre[b + 1] - 1]
                read = [g + b for g in range(g0, g1 + 1) if wbeg[g + 1] > wbeg[g]]
            assert written == read, (aligned, b)
        if aligned and E <= G:
            per_worker = np.bincount([g for (g, *_) in segs], minlength=G)
            assert per_worker.max() <= 1, "one partial per worker when the entries fit"


EDGE_CASES = [
    (74, 128, [4096] * 16),                 # DeepSeek-V3 batch: aligned, 8 vs 10 tile-times
    (74, 128, [131072] * 4),                # long context: aligned, 57 vs 59
    (74, 128, [0, 0, 0, 0, 0]),             # nothing to do
    (74, 128, [131072]),                    # one sequence over every worker
    (1, 64, [300, 5, 0, 77]),               # one worker
    (3, 64, [64, 64, 64]),                  # G == n
    (4, 64, [64, 65, 1]),                   # G == n + 1
    (100, 128, [1, 1, 1]),                  # far more workers than tiles
    (148, 64, [1, 63, 64, 65, 127, 128, 129, 1000]),
    (74, 128, [0, 127, 128, 129, 0, 255, 256, 257]),
    (16, 64, [5000, 17, 2222]),
]


def test_documented_plan_choices(harness):
    res = run_cases(harness, EDGE_CASES[:2])
    assert res[0]["aligned"] == 1 and res[0]["cost"] == 8 and res[0]["W"][-1] == 64
    assert res[1]["aligned"] == 1 and res[1]["cost"] == 57


def test_edge_cases(harness):
    for (G, tile, L), res in zip(EDGE_CASES, run_cases(harness, EDGE_CASES)):
        check_case(G, tile, L, res)


def test_random_batches(harness):
    rng = np.random.default_rng(2024)
    cases = []
    for i in range(400):
        B = int(rng.integers(1, 49))
        G = int(rng.integers(1, 201))
        tile = int(rng.choice([64, 128]))
        kind = i % 4
        if kind == 0:
            L = rng.integers(0, 9000, size=B)
        elif kind == 1:
            L = rng.integers(1, 200, size=B)
        elif kind == 2:
            L = np.full(B, int(rng.integers(1, 20000)))
        else:
            L = np.where(rng.random(B) < 0.3, 0, rng.integers(1024, 8193, size=B))
        cases.append((G, tile, [int(v) for v in L]))
    for (G, tile, L), res in zip(cases, run_cases(harness, cases)):
        check_case(G, tile, L, res)


def test_plan_choice_flips_for_many_ragged_sequences(harness):
    """Many short-and-long sequences: the even split wins (the aligned plan's
    longest entry exceeds the split's bound); the checks still hold."""
    rng = np.random.default_rng(7)
    L = [int(v) for v in rng.integers(1024, 8193, size=64)]
    (res,) = run_cases(harness, [(74, 128, L)])
    check_case(74, 128, L, res)
    assert res["aligned"] == 0

"""The C oracle against the brute-force restatement (tests/bruteforce.py) on
random tiny configurations: B in {1, 2, 3, 8}, pages of 2-4 rows, tails of
1-5 rows, up to 3 verify queries, duplicates, out-of-range rows, budget
overflows, admissions under capacity pressure with whole-request reclaim.

Agreement is required on return codes, location vectors, counters, hot-cache
tags and stamps, and optional page slots after every call.
"""
import numpy as np
import pytest

from bruteforce import BrutePool
from oracle import OraclePool


def _run_random(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 4))
    S = int(rng.integers(1, 3))
    T = int(rng.integers(1, 6))
    B = int(rng.choice([1, 2, 3, 8]))
    PR = int(rng.choice([2, 3, 4]))
    max_rows = 80
    cap = int(rng.integers(0, 30))
    reserve = int(rng.integers(0, min(cap, 3) + 1))
    E = 8
    orc = OraclePool(R, S, T, B, E, PR, max_rows, cap, reserve)
    bru = BrutePool(R, S, T, B, PR, cap, reserve)
    pages_max = -(-max_rows // PR)
    admitted = []
    for r in range(R):
        for s in range(S):
            N = int(rng.integers(0, 60))
            mask = (rng.random(N // PR) < 0.5).astype(np.uint8)
            a = orc.admit(r, s, N, mask, None)
            b = bru.admit(r, s, N, mask)
            assert a == tuple(b), (seed, "admit", r, s, a, b)
            if a[0] == "wouldwait":
                order = [int(x) for x in rng.permutation(R)]
                a2 = orc.reclaim(order, a[1])
                b2 = bru.reclaim(order, a[1])
                assert a2 == tuple(b2), (seed, "reclaim", a2, b2)
                a = orc.admit(r, s, N, mask, None)
                b = bru.admit(r, s, N, mask)
                assert a == tuple(b), (seed, "re-admit", a, b)
            if a[0] == 0:
                admitted.append((r, s))
            assert orc.used() == bru.used()
    for (r, s) in admitted:
        assert orc.state(r, s)[2].tolist() == bru.pages(r, s, pages_max)
    step = 0
    for _ in range(14):
        step += int(rng.integers(1, 3))  # steps may skip numbers
        for (r, s) in admitted:
            c = int(rng.integers(0, min(T, 2) + 1))
            L = orc.state(r, s)[3][1]
            if L + c <= max_rows:
                assert orc.append(r, s, c) == 0
                bru.append(r, s, c)
            L = orc.state(r, s)[3][1]
            Q = int(rng.integers(1, 4))
            k = int(rng.integers(0, 7))
            hi = L if rng.random() > 0.05 else L + 2
            if hi == 0:
                sel = np.zeros((Q, k), np.int32) - (1 if k else 0)
            else:
                sel = rng.integers(0, hi, size=(Q, k)).astype(np.int32)
            rc, loc, cnt = orc.resolve(step, r, s, sel)
            brc, bloc, bcnt = bru.resolve(step, r, s, sel.ravel().tolist())
            assert rc == brc, (seed, step, r, s, rc, brc)
            assert loc.ravel().tolist() == bloc, (seed, step, r, s)
            assert cnt.tolist() == bcnt, (seed, step, r, s, cnt, bcnt)
            tags, stamps, _, _ = orc.state(r, s)
            btags, bstamps = bru.tags(r, s)
            assert tags.tolist() == btags and stamps.tolist() == bstamps, (seed, step)
            assert orc.check(r, s) == 0
    return True


@pytest.mark.parametrize("block", range(8))
def test_oracle_matches_bruteforce(oracle_lib, block):
    for seed in range(block * 25, block * 25 + 25):
        assert _run_random(seed)

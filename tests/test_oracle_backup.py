"""Pins of the oracle's admission machinery beyond the hand-worked trace:
resident-first admission with deferred host backup, backup before a page
is freed, and bounded round-robin refill ("Adaptive DHiSparse", How it
works / Resident-first admission; Reclamation and refill).

  * random sequences of every admission, decode and resolution call on tiny
    pools: after each call the invariant that no row is without a copy
    (ready on the GPU or backed on the host) and the pool's bookkeeping
    hold, and every
    gathered row is the generator's payload of its row (a page freed
    without its backup, or refilled from a missing host copy, breaks it);
  * refill never takes the admission reserve;
  * round-robin closed form: k pages refilled from a cursor over R requests
    that each have enough missing pages give ceil(k/R) pages to the first
    k mod R requests visited and floor(k/R) to the rest.
"""
import numpy as np
import pytest

import dhs_workload
from oracle import OraclePool

TAG = 98  # RNG key of these payloads


def payload(r, s, row0, n, E):
    return dhs_workload.payload_rows(TAG, s, r, row0, n, E)


class Model:
    """Drives one oracle pool with random calls and checks it."""

    def __init__(self, rng, R=4, S=2, T=2, B=4, E=4, PR=4, max_rows=40, cap=10, reserve=1):
        self.rng = rng
        self.R, self.S, self.T, self.B, self.E, self.PR = R, S, T, B, E, PR
        self.max_rows, self.cap, self.reserve = max_rows, cap, reserve
        self.p = OraclePool(R, S, T, B, E, PR, max_rows, cap, reserve)
        self.L = {}
        self.step = 0

    def admitted(self):
        return sorted({r for (r, _) in self.L})

    def op(self):
        rng, R, S, E = self.rng, self.R, self.S, self.E
        kind = rng.choice(["admit", "admitdev", "append", "resolve", "reclaim",
                           "release", "backup", "refill"],
                          p=[.12, .18, .15, .25, .08, .06, .08, .08])
        if kind in ("admit", "admitdev"):
            r = int(rng.integers(R))
            if any(k[0] == r for k in self.L):
                return
            for s in range(S):
                N = int(rng.integers(0, self.max_rows - 8))
                pages = N // self.PR
                mask = (rng.random(pages) < 0.6).astype(np.uint8) if pages else None
                rows = payload(r, s, 0, N, E)
                fn = self.p.admit if kind == "admit" else self.p.admit_device
                rc, d = fn(r, s, N, mask, rows)
                if rc == "wouldwait":
                    others = [x for x in self.admitted() if x != r]
                    if self.p.reclaim(others, d)[0] == 0:
                        rc, d = fn(r, s, N, mask, rows)
                if rc == 0:
                    self.L[(r, s)] = N
        elif kind == "append":
            if not self.L:
                return
            r, s = list(self.L)[int(rng.integers(len(self.L)))]
            n = int(rng.integers(0, self.T + 1))
            n = min(n, self.max_rows - self.L[(r, s)])
            assert self.p.append(r, s, n, payload(r, s, self.L[(r, s)], n, E)) == 0
            self.L[(r, s)] += n
        elif kind == "resolve":
            if not self.L:
                return
            r, s = list(self.L)[int(rng.integers(len(self.L)))]
            L = self.L[(r, s)]
            if L == 0:
                return
            self.step += 1
            Q, k = int(rng.integers(1, 3)), int(rng.integers(1, 6))
            sel = rng.integers(0, L, size=(Q, k)).astype(np.int32)
            rc, loc, cnt = self.p.resolve(self.step, r, s, sel)
            if rc == 0:
                grc, st = self.p.gather(loc.ravel())
                assert grc == 0
                for e, row in enumerate(sel.ravel()):
                    assert np.array_equal(st[e], payload(r, s, int(row), 1, E)[0]), \
                        ("gathered row differs from payload", r, s, row)
            else:
                assert rc == "ebudget"
        elif kind == "reclaim":
            order = list(rng.permutation(self.R)[: int(rng.integers(1, self.R + 1))])
            self.p.reclaim(order, int(rng.integers(0, 6)))
        elif kind == "release":
            if not self.L:
                return
            r = self.admitted()[int(rng.integers(len(self.admitted())))]
            assert self.p.release(r) == 0
            for key in [k for k in self.L if k[0] == r]:
                del self.L[key]
        elif kind == "backup":
            assert self.p.backup(int(rng.integers(0, 5)))[0] == 0
        else:
            rc, n = self.p.refill(int(rng.integers(0, 6)))
            assert rc == 0
            assert self.p.used() <= self.cap - self.reserve

    def check(self):
        used = 0
        for r in range(self.R):
            for s in range(self.S):
                assert self.p.check(r, s) == 0, (r, s, self.p.check(r, s))
                used += int((self.p.state(r, s)[2] >= 0).sum())
        assert used == self.p.used() <= self.cap
        # every row of an admitted source: host copy valid unless its page is
        # resident (pending backup)
        for (r, s), L in self.L.items():
            pages = self.p.state(r, s)[2]
            host = self.p.rows(r, s, 0, 0, L)
            want = payload(r, s, 0, L, self.E)
            for row in range(L):
                q = row // self.PR
                if (q + 1) * self.PR <= L and pages[q] >= 0:
                    continue
                assert np.array_equal(host[row], want[row]), (r, s, row)


@pytest.mark.parametrize("seed", range(40))
def test_random_admission_sequences(oracle_lib, gen_lib, seed):
    m = Model(np.random.default_rng(seed), reserve=seed % 3)
    for _ in range(120):
        m.op()
        m.check()


def test_refill_keeps_the_reserve(oracle_lib):
    p = OraclePool(3, 1, 2, 2, 4, 4, 64, capacity=10, reserve=3)
    for r in range(3):
        assert p.admit(r, 0, 64, np.zeros(16, np.uint8), None) == (0, 0)
    rc, n = p.refill(100)
    assert rc == 0 and n == 7 and p.used() == 7


@pytest.mark.parametrize("k", [0, 1, 2, 5, 7, 11])
def test_round_robin_closed_form(oracle_lib, k):
    R, pages = 4, 8
    p = OraclePool(R, 1, 2, 2, 4, 4, 32, capacity=64, reserve=0)
    for r in range(R):
        assert p.admit(r, 0, pages * 4, np.zeros(pages, np.uint8), None) == (0, 0)
    # move the cursor to request 2 first: 2 pages from a cursor of 0
    assert p.refill(2) == (0, 2)
    before = np.array([(p.state(r, 0)[2] >= 0).sum() for r in range(R)])
    assert p.refill(k) == (0, k)
    got = np.array([(p.state(r, 0)[2] >= 0).sum() for r in range(R)]) - before
    order = [2, 3, 0, 1]  # visit order from the cursor
    want = np.zeros(R, int)
    for i, r in enumerate(order):
        want[r] = k // R + (1 if i < k % R else 0)
    assert np.array_equal(got, want), (got, want)


@pytest.mark.parametrize("seed", range(6))
def test_lockstep_driver_on_the_oracle(oracle_lib, gen_lib, seed):
    """The lockstep driver the GPU parity test uses, run on the oracle alone
    (its own checks: bookkeeping, host rows, payload bytes)."""
    from admission_seq import run_sequence
    from fixture_runner import OracleAdapter
    run_sequence([OracleAdapter()], seed, reserve=seed % 3)

"""Random sequences of admission, backup, refill, decode and resolution
calls, run in lockstep on several implementations (adapters with the
interface of fixture_runner.OracleAdapter) and compared call by call.

Every gathered row must also be the generator's payload of its row, so a
page freed before its backup, or refilled from a host copy that was never
written, shows up as wrong bytes even where both sides agree."""
from __future__ import annotations

import numpy as np

import dhs_workload

TAG = 99  # RNG key of these payloads


def payload(r, s, row0, n, E):
    return dhs_workload.payload_rows(TAG, s, r, row0, n, E)


def run_sequence(apis, seed, n_ops=80, R=4, S=2, T=2, B=4, E=8, PR=4, max_rows=40,
                 cap=10, reserve=1, max_q=3, max_k=6):
    rng = np.random.default_rng(seed)
    for a in apis:
        a.new_pool(R, S, T, B, E, PR, max_rows, cap, reserve)
    L = {}
    step = 0

    def same(vals, what):
        for v in vals[1:]:
            if isinstance(v, np.ndarray) or isinstance(vals[0], np.ndarray):
                assert np.array_equal(np.asarray(v), np.asarray(vals[0])), (seed, what, vals)
            else:
                assert v == vals[0], (seed, what, vals)
        return vals[0]

    for i in range(n_ops):
        kind = rng.choice(["admit", "admitdev", "append", "resolve", "reclaim",
                           "release", "backup", "refill"],
                          p=[.12, .18, .15, .25, .08, .06, .08, .08])
        admitted = sorted({r for (r, _) in L})
        if kind in ("admit", "admitdev"):
            r = int(rng.integers(R))
            if r in admitted:
                continue
            for s in range(S):
                N = int(rng.integers(0, max_rows - 8))
                pages = N // PR
                mask = (rng.random(pages) < 0.6).astype(np.uint8) if pages else None
                rows = payload(r, s, 0, N, E)
                fn = "admit" if kind == "admit" else "admit_device"
                rc, d = same([getattr(a, fn)(r, s, N, mask, rows) for a in apis], (i, fn))
                if rc == "wouldwait":
                    others = [x for x in admitted if x != r]
                    rc2 = same([a.reclaim(others, d) for a in apis], (i, "reclaim"))
                    if rc2[0] == 0:
                        rc, d = same([getattr(a, fn)(r, s, N, mask, rows) for a in apis],
                                     (i, fn))
                if rc == 0:
                    L[(r, s)] = N
        elif kind == "append" and L:
            r, s = list(L)[int(rng.integers(len(L)))]
            n = min(int(rng.integers(0, T + 1)), max_rows - L[(r, s)])
            rows = payload(r, s, L[(r, s)], n, E)
            same([a.append(r, s, n, rows) for a in apis], (i, "append"))
            L[(r, s)] += n
        elif kind == "resolve" and L:
            r, s = list(L)[int(rng.integers(len(L)))]
            if L[(r, s)] == 0:
                continue
            step += 1
            Q, k = int(rng.integers(1, max_q + 1)), int(rng.integers(1, max_k + 1))
            sel = rng.integers(0, L[(r, s)], size=(Q, k)).astype(np.int32)
            outs = [a.resolve(step, r, s, sel) for a in apis]
            rc = same([o[0] for o in outs], (i, "resolve rc"))
            same([np.asarray(o[1]).ravel() for o in outs], (i, "loc"))
            same([np.asarray(o[2]) for o in outs], (i, "counters"))
            if rc == 0:
                for a in apis:
                    st = np.asarray(a.gather(np.asarray(outs[0][1]).ravel()))
                    for e, row in enumerate(sel.ravel()):
                        assert np.array_equal(st[e], payload(r, s, int(row), 1, E)[0]), \
                            (seed, i, type(a).__name__, r, s, int(row))
        elif kind == "reclaim":
            order = [int(x) for x in rng.permutation(R)[: int(rng.integers(1, R + 1))]]
            deficit = int(rng.integers(0, 6))
            same([a.reclaim(order, deficit) for a in apis], (i, "reclaim"))
        elif kind == "release" and admitted:
            r = admitted[int(rng.integers(len(admitted)))]
            same([a.release(r) for a in apis], (i, "release"))
            for key in [k for k in L if k[0] == r]:
                del L[key]
        elif kind == "backup":
            n = int(rng.integers(0, 5))  # one draw for every implementation
            same([a.backup(n) for a in apis], (i, "backup"))
        elif kind == "refill":
            n = int(rng.integers(0, 6))
            same([a.refill(n) for a in apis], (i, "refill"))
        # bookkeeping after every call
        same([a.used() for a in apis], (i, "used"))
        same([a.pending_backup() for a in apis], (i, "pending"))
        for (r, s), n in L.items():
            pages = same([np.asarray(a.pages(r, s)) for a in apis], (i, "pages", r, s))
            want = payload(r, s, 0, n, E)
            for a in apis:
                host = a.host_rows(r, s, 0, n)
                for row in range(n):
                    q = row // PR
                    if (q + 1) * PR <= n and pages[q] >= 0:
                        continue  # resident: its backup may still be deferred
                    assert np.array_equal(host[row], want[row]), \
                        (seed, i, type(a).__name__, r, s, row)

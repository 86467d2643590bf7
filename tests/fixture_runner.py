"""Parser and runner for the hand-worked traces under tests/golden.

A trace is a list of commands (pool, admit, admitdev, admitwin, backup,
refill, pending, hostok, reclaim, release, used, pages, append, resolve) each
followed by the values worked out by hand.  The runner
drives any implementation through a small adapter (the oracle, or the CUDA
library through its C ABI) and checks every expected value, plus byte truth:
each gathered row of a successful resolve equals the generator's payload of
the selected row.
"""
from __future__ import annotations

import os

import numpy as np

import dhs_workload

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
PAYLOAD_TAG = 97  # RNG key of the trace payloads


def parse(name: str):
    cmds = []
    with open(os.path.join(GOLDEN, name)) as f:
        for ln, line in enumerate(f, 1):
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            cmds.append((ln, line.split()))
    return cmds


def _loc_token(tok: str) -> int:
    if tok == "X":
        return 0xFFFFFFFF
    tier = {"T": 0, "O": 1, "H": 2}[tok[0]]
    return (tier << 30) | int(tok[1:])


def _rc(tok: str):
    return 0 if tok == "ok" else tok


def run_trace(name: str, api, elems: int | None = None):
    """Run one golden trace against `api`; raises AssertionError on the
    first mismatch (message names the trace line)."""
    cmds = parse(name)
    E = None
    last = None  # (rc, loc, counters, sel, r, s)
    lengths = {}
    for ln, tok in cmds:
        where = f"{name}:{ln}"
        op = tok[0]
        if op == "pool":
            R, S, T, B, E0, PR, max_rows, cap, reserve = map(int, tok[1:10])
            tail_rows = T
            E = elems or E0
            api.new_pool(R, S, T, B, E, PR, max_rows, cap, reserve)
        elif op == "admit":
            r, s, N = map(int, tok[1:4])
            m = tok[4]
            mask = None if m == "*" else np.array([int(c) for c in m], np.uint8)
            host = dhs_workload.payload_rows(PAYLOAD_TAG, s, r, 0, N, E)
            rc, deficit = api.admit(r, s, N, mask, host)
            assert tok[5] == "->"
            assert rc == _rc(tok[6]), f"{where}: rc {rc} != {tok[6]}"
            assert deficit == int(tok[7]), f"{where}: deficit {deficit} != {tok[7]}"
            if rc == 0:
                lengths[(r, s)] = N
        elif op == "admitdev":
            r, s, N = map(int, tok[1:4])
            m = tok[4]
            mask = None if m == "*" else np.array([int(c) for c in m], np.uint8)
            rows = dhs_workload.payload_rows(PAYLOAD_TAG, s, r, 0, N, E)
            rc, deficit = api.admit_device(r, s, N, mask, rows)
            assert tok[5] == "->"
            assert rc == _rc(tok[6]), f"{where}: rc {rc} != {tok[6]}"
            assert deficit == int(tok[7]), f"{where}: deficit {deficit} != {tok[7]}"
            if rc == 0:
                lengths[(r, s)] = N
        elif op == "admitwin":
            r, s, N = map(int, tok[1:4])
            m = min(N, tail_rows)
            rows = dhs_workload.payload_rows(PAYLOAD_TAG, s, r, N - m, m, E)
            rc = api.admit_window(r, s, N, rows)
            assert tok[4] == "->"
            assert rc == _rc(tok[5]), f"{where}: rc {rc} != {tok[5]}"
            if rc == 0:
                lengths[(r, s)] = N
        elif op in ("backup", "refill"):
            rc, n = getattr(api, op)(int(tok[1]))
            assert tok[2] == "->"
            assert rc == _rc(tok[3]), f"{where}: rc {rc} != {tok[3]}"
            assert n == int(tok[4]), f"{where}: {op} {n} != {tok[4]}"
        elif op == "pending":
            got = api.pending_backup()
            assert got == int(tok[1]), f"{where}: pending {got} != {tok[1]}"
        elif op == "hostok":
            r, s, row0, n = map(int, tok[1:5])
            got = api.host_rows(r, s, row0, n)
            want = dhs_workload.payload_rows(PAYLOAD_TAG, s, r, row0, n, E)
            assert np.array_equal(got, want), f"{where}: host rows differ from payload"
        elif op == "reclaim":
            order = [] if tok[1] == "-" else [int(x) for x in tok[1].split(",")]
            rc, freed = api.reclaim(order, int(tok[2]))
            assert rc == _rc(tok[4]), f"{where}: rc {rc} != {tok[4]}"
            assert freed == int(tok[5]), f"{where}: freed {freed} != {tok[5]}"
        elif op == "release":
            r = int(tok[1])
            rc = api.release(r)
            assert rc == _rc(tok[3]), f"{where}: rc {rc}"
            for key in [k for k in lengths if k[0] == r]:
                del lengths[key]
        elif op == "used":
            assert api.used() == int(tok[1]), f"{where}: used {api.used()} != {tok[1]}"
        elif op == "pages":
            r, s = int(tok[1]), int(tok[2])
            want = np.array([int(x) for x in tok[4:]], np.int32)
            got = api.pages(r, s)[: len(want)]
            assert np.array_equal(got, want), f"{where}: pages {got} != {want}"
        elif op == "append":
            r, s, count = map(int, tok[1:4])
            L = lengths[(r, s)]
            rows = dhs_workload.payload_rows(PAYLOAD_TAG, s, r, L, count, E)
            rc = api.append(r, s, count, rows)
            assert rc == 0, f"{where}: append rc {rc}"
            lengths[(r, s)] = L + count
        elif op == "resolve":
            step, r, s, Q, k = map(int, tok[1:6])
            assert tok[6] == ":"
            sel = np.array([int(x) for x in tok[7: 7 + Q * k]], np.int32).reshape(Q, k)
            assert tok[7 + Q * k] == "->"
            want_rc = _rc(tok[8 + Q * k])
            rc, loc, cnt = api.resolve(step, r, s, sel)
            assert rc == want_rc, f"{where}: rc {rc} != {want_rc}"
            last = (rc, np.asarray(loc).ravel(), np.asarray(cnt), sel, r, s)
            if rc == 0:
                # byte truth: every gathered row is the selected row's payload
                staging = np.asarray(api.gather(np.asarray(loc).ravel()))
                for e, row in enumerate(sel.ravel()):
                    want = dhs_workload.payload_row(PAYLOAD_TAG, s, r, int(row), E)
                    assert np.array_equal(staging[e], want), \
                        f"{where}: staging row {e} (row {row}) differs from payload"
        elif op == "loc":
            want = np.array([_loc_token(t) for t in tok[1:]], np.uint32)
            assert np.array_equal(last[1], want), f"{where}: loc {last[1]} != {want}"
        elif op == "counters":
            want = np.array([int(t) for t in tok[1:]], np.uint32)
            assert np.array_equal(last[2], want), f"{where}: counters {last[2]} != {want}"
        elif op in ("tags", "stamps"):
            r, s = int(tok[1]), int(tok[2])
            want = np.array([int(t) for t in tok[4:]], np.int64)
            tags, stamps = api.state(r, s)
            got = np.asarray(tags if op == "tags" else stamps, np.int64)
            assert np.array_equal(got, want), f"{where}: {op} {got} != {want}"
        else:
            raise ValueError(f"{where}: unknown command {op}")


class OracleAdapter:
    """Drives the CPU oracle."""

    def new_pool(self, R, S, T, B, E, PR, max_rows, cap, reserve):
        from oracle import OraclePool
        self.p = OraclePool(R, S, T, B, E, PR, max_rows, cap, reserve)

    def admit(self, r, s, N, mask, host):
        return self.p.admit(r, s, N, mask, host)

    def admit_device(self, r, s, N, mask, rows):
        return self.p.admit_device(r, s, N, mask, rows)

    def admit_window(self, r, s, N, rows):
        return self.p.admit_window(r, s, N, rows)

    def backup(self, n):
        return self.p.backup(n)

    def refill(self, n):
        return self.p.refill(n)

    def pending_backup(self):
        return self.p.pending_backup()

    def host_rows(self, r, s, row0, n):
        return self.p.rows(r, s, 0, row0, n)

    def reclaim(self, order, deficit):
        return self.p.reclaim(order, deficit)

    def release(self, r):
        return self.p.release(r)

    def used(self):
        return self.p.used()

    def pages(self, r, s):
        return self.p.state(r, s)[2]

    def append(self, r, s, count, rows):
        return self.p.append(r, s, count, rows)

    def resolve(self, step, r, s, sel):
        return self.p.resolve(step, r, s, sel)

    def gather(self, loc):
        rc, st = self.p.gather(loc)
        assert rc == 0
        return st

    def state(self, r, s):
        t, st, _, _ = self.p.state(r, s)
        return t, st

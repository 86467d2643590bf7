"""Brute-force restatement of resolution, for tiny inputs only.

Independent of the C oracle in formulation: Python sets and dicts, the
optional slot allocator as "min of the free set", step-1 membership by set
lookups, the hot cache as a row -> slot dictionary, and LRU in its batched
form -- all unprotected slots sorted by (last use, slot) and the first m
given to the m missing rows in ascending order -- where the oracle evicts
one victim at a time with a linear scan.  The two agree only if the batched
and sequential statements of LRU agree.
"""
from __future__ import annotations

NO_LOC = 0xFFFFFFFF


def _loc(tier, idx):
    return (tier << 30) | idx


class BrutePool:
    def __init__(self, R, S, T, B, PR, capacity, reserve=0):
        self.R, self.S, self.T, self.B, self.PR = R, S, T, B, PR
        self.free = set(range(capacity))
        self.capacity, self.reserve = capacity, reserve
        self.src = {}

    def used(self):
        return self.capacity - len(self.free)

    def admit(self, r, s, N, mask):
        if (r, s) in self.src:
            return "estate", 0
        complete = N // self.PR
        pages = [p for p in range(complete) if mask is None or mask[p]]
        if self.used() + len(pages) > self.capacity - self.reserve:
            return "wouldwait", self.used() + len(pages) - (self.capacity - self.reserve)
        ready = {}
        for p in pages:
            slot = min(self.free)
            self.free.remove(slot)
            ready[p] = slot
        self.src[(r, s)] = {
            "N": N, "L": N, "ready": ready, "cache": {},
            "slot_row": [None] * self.B, "last_use": [0] * self.B}
        return 0, 0

    def reclaim(self, order, deficit):
        seen, avail = set(), 0
        for r in order:
            if r not in seen:
                seen.add(r)
                avail += sum(len(st["ready"]) for (rr, _), st in self.src.items() if rr == r)
        if avail < deficit:
            return "wouldwait", 0
        got = 0
        for r in order:
            if got >= deficit:
                break
            for (rr, _), st in self.src.items():
                if rr == r:
                    for slot in st["ready"].values():
                        self.free.add(slot)
                        got += 1
                    st["ready"] = {}
        return 0, got

    def append(self, r, s, count):
        self.src[(r, s)]["L"] += count
        return 0

    def resolve(self, step, r, s, sel_rows):
        """sel_rows: flat list of Q*k rows.  Returns (rc, loc list, counters)."""
        st = self.src[(r, s)]
        pair = r * self.S + s
        L, N, T, B, PR = st["L"], st["N"], self.T, self.B, self.PR
        n = len(sel_rows)
        tail_rows = set(range(max(0, L - T), L))

        def step1_only():  # a failed step: locations of what step 1 holds
            out = []
            for row in sel_rows:
                if row in tail_rows:
                    out.append(_loc(0, pair * T + row % T))
                elif 0 <= row < L and row // PR in st["ready"] and (row // PR + 1) * PR <= N:
                    out.append(_loc(1, st["ready"][row // PR] * PR + row % PR))
                else:
                    out.append(NO_LOC)
            return out

        if any(x < 0 or x >= L for x in sel_rows):
            return "erange", step1_only(), [0] * 8
        union = sorted(set(sel_rows))
        where, pending, touched = {}, [], set()
        c = dict(tail=0, opt=0, hot=0, host=0, scan=0, ev=0)
        for row in union:
            page = row // PR
            if row in tail_rows:
                where[row] = _loc(0, pair * T + row % T)
                c["tail"] += 1
            elif page in st["ready"] and (page + 1) * PR <= N:
                where[row] = _loc(1, st["ready"][page] * PR + row % PR)
                c["opt"] += 1
            elif row in st["cache"]:
                j = st["cache"][row]
                touched.add(j)
                where[row] = _loc(2, pair * B + j)
                c["hot"] += 1
                c["scan"] = max(c["scan"], j + 1)
            else:
                pending.append(row)
                c["scan"] = B
        use = [step if j in touched else st["last_use"][j] for j in range(B)]
        free = sorted((use[j], j) for j in range(B) if use[j] != step)
        if len(pending) > len(free):
            return "ebudget", step1_only(), [0] * 8
        for row, (_, j) in zip(pending, free):
            old = st["slot_row"][j]
            if old is not None:
                del st["cache"][old]
                c["ev"] += 1
            st["slot_row"][j] = row
            st["cache"][row] = j
            use[j] = step
            where[row] = _loc(2, pair * B + j)
            c["host"] += 1
        st["last_use"] = use
        counters = [n, len(union), c["tail"], c["opt"], c["hot"], c["host"],
                    c["scan"], c["ev"]]
        return 0, [where[x] for x in sel_rows], counters

    def tags(self, r, s):
        st = self.src[(r, s)]
        return [-1 if x is None else x for x in st["slot_row"]], list(st["last_use"])

    def pages(self, r, s, pages_max):
        st = self.src[(r, s)]
        return [st["ready"].get(p, -1) for p in range(pages_max)]

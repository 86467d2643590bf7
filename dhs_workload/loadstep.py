"""Load-step workload: admission pressure rising and draining.

"Adaptive DHiSparse", Evidence (load-step on/off experiment): with optional
residency on, fewer selected rows come from the host while load is low; the
optional pages give way when admissions need memory and come back once the
extra requests have left.  The pages give no schedule,
model or sizes for it; this recipe stands in with three phases over one
pool whose optional capacity holds `low` requests' histories:

  low    steps [1, steps_low]: requests 0 .. low-1 arrive at step 1;
  burst  requests low .. slots-1 arrive at step steps_low + 1, each
         admitted resident-first, reclaiming whole older requests (oldest
         first) to cover its deficit;
  drain  the burst requests finish at step steps_low + steps_burst + 1;
         requests 0 .. low-1 remain and refill their pages.

Every step: departures, arrivals, then (residency on) a bounded refill and
a bounded host backup, then each active (request, source) appends one
decode row and resolves k rows.  Selections follow the other workloads'
recipe (recency window + Zipf over the imported history, temporal locality
rho), keyed by (request, source, the request's own step).  With residency
off the pool has no optional capacity: every imported row comes from the
hot cache or the host.

This module only draws inputs; `run` drives any implementation through an
adapter with the interface of the tests' OracleAdapter (plus, optionally,
`decode_step(step, work)` running a whole step's appends and resolves as
one batch).
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import SEED, payload_rows, permutation, select, zipf_cdf


@dataclasses.dataclass(frozen=True)
class LoadStepConfig:
    name: str
    tag: int
    slots: int              # request slots (the burst fills all of them)
    low: int                # requests at low load (their pages fit)
    sources: int
    history: int            # imported rows per (request, source)
    tail: int
    hot: int
    topk: int
    steps_low: int
    steps_burst: int
    steps_drain: int
    refill_per_step: int
    backup_per_step: int
    rho: float = 0.9
    window: int = 1024
    frac_recent: float = 0.7
    zipf_s: float = 1.1
    row_elems: int = 576
    page_rows: int = 64

    @property
    def total_steps(self) -> int:
        return self.steps_low + self.steps_burst + self.steps_drain

    @property
    def max_rows(self) -> int:
        return self.history + self.total_steps

    @property
    def pages_per_request(self) -> int:
        return self.sources * (self.history // self.page_rows)

    @property
    def capacity(self) -> int:
        """Optional pages: exactly the low-load requests' histories."""
        return self.low * self.pages_per_request

    def phase(self, step: int) -> str:
        if step <= self.steps_low:
            return "low"
        if step <= self.steps_low + self.steps_burst:
            return "burst"
        return "drain"

    def arrivals(self, step: int) -> list[int]:
        if step == 1:
            return list(range(self.low))
        if step == self.steps_low + 1:
            return list(range(self.low, self.slots))
        return []

    def departures(self, step: int) -> list[int]:
        if step == self.steps_low + self.steps_burst + 1:
            return list(range(self.low, self.slots))
        return []

    def arrival_step(self, r: int) -> int:
        return 1 if r < self.low else self.steps_low + 1


# small enough for the oracle and the parity tests
LOADSTEP_SMALL = LoadStepConfig(
    name="loadstep_small", tag=21, slots=12, low=3, sources=1, history=2048, tail=16,
    hot=96, topk=96, steps_low=6, steps_burst=8, steps_drain=10, refill_per_step=16,
    backup_per_step=8, window=64, row_elems=64)

# the measured run: 32 slots, 8 of them at low load, 2 KV sources of 16K rows
LOADSTEP = LoadStepConfig(
    name="loadstep", tag=22, slots=32, low=8, sources=2, history=16384, tail=256,
    hot=2048, topk=1024, steps_low=16, steps_burst=32, steps_drain=32,
    refill_per_step=128, backup_per_step=128)


class LoadStepInputs:
    """Seeded inputs: payload rows and per-step selections."""

    def __init__(self, cfg: LoadStepConfig, seed: int = SEED):
        self.cfg = cfg
        self.seed = seed
        self._cdf = zipf_cdf(cfg.history, cfg.zipf_s)
        self._perm = {}
        self._prev = {}

    def rows(self, r: int, s: int, row0: int, n: int) -> np.ndarray:
        return payload_rows(self.cfg.tag, s, r, row0, n, self.cfg.row_elems, self.seed)

    def selection(self, r: int, s: int, local_step: int, L: int) -> np.ndarray:
        """k distinct rows of [0, L) for the request's local_step-th step
        (call in step order per (r, s): temporal locality keeps state)."""
        c = self.cfg
        key = (r, s)
        if key not in self._perm:
            self._perm[key] = permutation(c.tag, s, r, c.history, self.seed)
        if local_step == 1:
            self._prev[key] = None
        rows, z = select(c.tag, s, r, local_step, 0, L, c.history, c.topk, c.window,
                         c.frac_recent, self._cdf, self._perm[key], self._prev[key],
                         c.rho, None, self.seed)
        self._prev[key] = z
        return rows


def run(api, cfg: LoadStepConfig, residency: bool = True, inputs=None, on_step=None):
    """Drive `api` through the load-step schedule.  Returns one record per
    step: {"step", "phase", "active", "unique", "host", "resident_pages",
    "pending_backup"} with the tier counters summed over the step's
    resolves.  `on_step(step, results)` sees each step's per-item results
    [(r, s, rc, loc, counters, sel)]."""
    c = cfg
    inputs = inputs or LoadStepInputs(c)
    api.new_pool(c.slots, c.sources, c.tail, c.hot, c.row_elems, c.page_rows, c.max_rows,
                 c.capacity if residency else 0, 0)
    active: dict[int, int] = {}  # request -> rows appended so far
    order: list[int] = []        # admitted requests, oldest first
    records = []
    pages = c.history // c.page_rows
    for step in range(1, c.total_steps + 1):
        for r in c.departures(step):
            assert api.release(r) == 0
            del active[r]
            order.remove(r)
        for r in c.arrivals(step):
            for s in range(c.sources):
                mask = None if residency else np.zeros(pages, np.uint8)
                rows = inputs.rows(r, s, 0, c.history)
                rc, d = api.admit_device(r, s, c.history, mask, rows)
                if rc == "wouldwait":  # reclaim whole older requests, oldest first
                    rc2, _ = api.reclaim([x for x in order if x != r], d)
                    assert rc2 == 0, (step, r, rc2)
                    rc, d = api.admit_device(r, s, c.history, mask, rows)
                assert rc == 0, (step, r, s, rc)
            active[r] = 0
            order.append(r)
        if residency:
            assert api.refill(c.refill_per_step)[0] == 0
            assert api.backup(c.backup_per_step)[0] == 0
        work = []  # (r, s, appended row, selection)
        for r in sorted(active):
            local = step - c.arrival_step(r) + 1
            L = c.history + active[r]
            active[r] += 1
            for s in range(c.sources):
                work.append((r, s, inputs.rows(r, s, L, 1),
                             inputs.selection(r, s, local, L + 1)))
        if hasattr(api, "decode_step"):  # one batched decode step
            outs = api.decode_step(step, work)
        else:
            outs = []
            for r, s, row, _ in work:
                assert api.append(r, s, 1, row) == 0
            for r, s, _, sel in work:
                outs.append(api.resolve(step, r, s, sel[None]))
        results = [(r, s, rc, loc, cnt, sel)
                   for (r, s, _, sel), (rc, loc, cnt) in zip(work, outs)]
        if on_step:
            on_step(step, results)
        cnt = np.array([x[4] for x in results], np.int64)
        records.append({"step": step, "phase": c.phase(step), "active": len(active),
                        "unique": int(cnt[:, 1].sum()), "host": int(cnt[:, 5].sum()),
                        "resident_pages": int(api.used()),
                        "pending_backup": int(api.pending_backup())})
    return records


def phase_fractions(records) -> dict:
    """Host-fetched fraction of unique selected rows per phase."""
    out = {}
    for ph in ("low", "burst", "drain"):
        rs = [x for x in records if x["phase"] == ph]
        u = sum(x["unique"] for x in rs)
        out[ph] = sum(x["host"] for x in rs) / u if u else 0.0
    return out

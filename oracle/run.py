"""Drive the oracle through a whole synthetic workload.

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline).

Per step s of a configuration, for every simulated request r:
  1. every source appends its step-s decode rows (tail ring + host copy);
  2. every source resolves its selection for the step (all Q verify
     queries at once);
  3. one gather per layer: the S resolving layers gather their own location
     vectors, then `reuse_layers` Reuse layers gather source 0's location
     vector again ("Model-specific reuse": they inherit it, no resolution).

With union=True every source resolves in the union staging layout (each
distinct row of a verify block staged once, plus per-query index lists) and
each layer gathers the U union rows only.

Admission runs for every request (page slots depend on admission order), but
only the simulated requests hold row bytes and are stepped; requests are
independent once admitted, so a sampled subset gives exact per-request
results for the full-size workload.
"""
from __future__ import annotations

import numpy as np

from dhs_workload.configs import Config, Workload, drive_admission

from . import OraclePool


class _AdmitAdapter:
    def __init__(self, run):
        self.run = run

    def admit(self, r, s, mask):
        return self.run.admit(r, s, mask)

    def reclaim(self, order, deficit):
        return self.run.pool.reclaim(order, deficit)


class OracleRun:
    def __init__(self, cfg: Config, wl: Workload | None = None,
                 requests=None, payload: bool = True, capacity=None,
                 union: bool = False):
        self.cfg = cfg
        self.union = union
        self.wl = wl or Workload(cfg)
        self.requests = list(range(cfg.requests)) if requests is None else list(requests)
        self.payload = payload
        self._cap = cfg.pool_pages() if capacity is None else capacity
        self._sim = set(self.requests)
        self._host = {}
        self.reset()

    def reset(self):
        """A fresh pool with every request admitted again (row bytes of the
        simulated requests are generated once and kept)."""
        cfg = self.cfg
        if getattr(self, "pool", None) is not None:
            self.pool.close()
        self.pool = OraclePool(cfg.requests, cfg.sources, cfg.tail, cfg.hot,
                               cfg.row_elems, cfg.page_rows, cfg.max_rows, self._cap)
        drive_admission(_AdmitAdapter(self), cfg, self.wl)

    def admit(self, r, s, mask):
        host = None
        if self.payload and r in self._sim:
            host = self._host.get((r, s))
            if host is None:
                host = np.empty((self.cfg.history, self.cfg.row_elems), np.uint16)
                self.wl.fill_host_rows(host.ctypes.data, self.cfg.history, [(r, s)])
                self._host[(r, s)] = host
        return self.pool.admit(r, s, self.cfg.history, mask, host)

    def layers(self):
        """(kind, source) per layer of a request, in staging order."""
        c = self.cfg
        return ([("resolve", s) for s in range(c.sources)]
                + [("reuse", 0)] * c.reuse_layers)

    def step(self, step: int, gather: bool = True):
        """Run one step; returns {r: {"rc": [S], "loc": [S][Q][k],
        "counters": [S][8], "staging": [layers][Q][k][E] or None}}.
        Union layout: "loc" is [S][Q*k] (U union locations, then END_LOC),
        "index" [S][Q][k], and "staging" a list of [U][E] arrays per layer."""
        c = self.cfg
        out = {}
        pairs = [(r, s) for r in self.requests for s in range(c.sources)]
        counts, rows = self.wl.appended_rows(step, pairs) if self.payload else (
            np.array([self.wl.append[r, step - 1] for (r, _) in pairs]), None)
        for i, (r, s) in enumerate(pairs):
            rc = self.pool.append(r, s, int(counts[i]),
                                  rows[i, : counts[i]] if rows is not None else None)
            if rc != 0:
                raise RuntimeError(f"oracle append failed: {rc}")
        for r in self.requests:
            rcs, locs, cnts, idxs = [], [], [], []
            for s in range(c.sources):
                sel = self.wl.sel(step, r, s)
                if self.union:
                    rc, loc, idx, cnt = self.pool.resolve_union(step, r, s, sel)
                    idxs.append(idx)
                else:
                    rc, loc, cnt = self.pool.resolve(step, r, s, sel)
                rcs.append(rc)
                locs.append(loc)
                cnts.append(cnt)
            res = {"rc": rcs, "loc": np.stack(locs), "counters": np.stack(cnts),
                   "staging": None}
            if self.union:
                res["index"] = np.stack(idxs)
            if gather and self.payload:
                st = []
                for kind, s in self.layers():
                    want = locs[s][: int(cnts[s][1])] if self.union else locs[s]
                    rc, g = self.pool.gather(want)
                    if rc != 0:
                        raise RuntimeError(f"oracle gather failed: {rc}")
                    st.append(g)
                res["staging"] = st if self.union else np.stack(st)
            out[r] = res
        return out

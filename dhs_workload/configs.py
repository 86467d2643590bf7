"""The five synthetic workloads and their seeded inputs.

Shapes follow the configurations named for the path (histories of 32K-500K
rows of 576 bf16, concurrency 8-128, an 8-query verify block, layer reuse);
"K" is read as 1024 rows (32K = 32768, 100K = 102400, 500K = 512000).
Everything here is input preparation: which rows a step selects, which
pages start optional-resident, how many rows each step appends, and the row
bytes.  Nothing here resolves, evicts or gathers.

Selection recipe (per request, source and step; k distinct rows):
  * min(round(0.7 k), W) rows uniform without replacement from the recency
    window [L - W, L), W = min(1024, L) -- for k = 2048 the whole window;
  * the rest distinct Zipf(s = 1.1) draws over the imported history [0, N),
    ranks mapped to rows by a seeded per-(request, source) permutation;
  * with temporal locality rho > 0, each previous-step Zipf row is first kept
    with probability rho;
  * a verify block of Q queries shares a core of `verify_core` rows and adds
    k - core query-specific rows per query (pairwise overlap core / k);
  * sorted ascending.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os

import numpy as np

from . import (SEED, append_counts, payload_pairs_into, permutation,
               residency, select, zipf_cdf)


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    tag: int                      # RNG key of the workload
    requests: int                 # R
    sources: int                  # KV sources per request with own state+payload
    history: int                  # N imported rows per (request, source)
    tail: int                     # T rows of mutable tail
    hot: int                      # B hot-cache rows
    topk: int                     # k selected rows per query
    queries: int = 1              # Q verify queries per step
    steps: int = 16               # timed steps
    warmup_steps: int = 0         # steps run before the timed ones
    residency: float | None = 0.5  # resident fraction of complete pages
    capacity_frac: float | None = None  # admission-driven: pool = frac * pages
    append_lo: int = 1            # rows appended per request per step: U[lo, hi]
    append_hi: int = 1
    reuse_layers: int = 0         # gather-only layers reusing source 0's locations
    shared_selection: bool = False  # all sources use source 0's selection
    rho: float = 0.0              # temporal locality of the Zipf part
    verify_core: int = 0          # rows shared by all verify queries
    window: int = 1024
    frac_recent: float = 0.7
    zipf_s: float = 1.1
    row_elems: int = 576
    page_rows: int = 64

    @property
    def row_bytes(self) -> int:
        return self.row_elems * 2

    @property
    def total_steps(self) -> int:
        return self.warmup_steps + self.steps

    @property
    def max_rows(self) -> int:
        return self.history + self.total_steps * self.append_hi

    @property
    def complete_pages(self) -> int:
        return self.history // self.page_rows

    @property
    def pages_max(self) -> int:
        return -(-self.max_rows // self.page_rows)

    @property
    def pairs(self) -> int:
        return self.requests * self.sources

    @property
    def layers(self) -> int:
        """Gathers per request per step (resolving layers + reuse layers)."""
        return self.sources + self.reuse_layers

    @property
    def entries_per_step(self) -> int:
        """Selected rows gathered into staging per step."""
        return self.requests * self.layers * self.queries * self.topk

    @property
    def resolved_per_step(self) -> int:
        return self.requests * self.sources * self.queries * self.topk

    def resident_pages(self) -> int:
        """Resident complete pages per (request, source), fixed residency."""
        assert self.residency is not None
        return int(round(self.residency * self.complete_pages))

    def pool_pages(self) -> int:
        """Optional-pool capacity in pages."""
        if self.capacity_frac is not None:
            return int(round(self.capacity_frac * self.pairs * self.complete_pages))
        return self.pairs * self.resident_pages()

    def scaled(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


TINY = Config("tiny", 1, requests=1, sources=1, history=4096, tail=64, hot=512,
              topk=256, steps=16, residency=0.5)
C8 = Config("c8", 2, requests=8, sources=4, history=32768, tail=256, hot=4096,
            topk=2048, steps=64, residency=1.0)
C64 = Config("c64", 3, requests=64, sources=4, history=32768, tail=256,
             hot=4096, topk=2048, queries=8, verify_core=1638, steps=32,
             residency=0.4, append_lo=1, append_hi=8)
C128 = Config("c128", 4, requests=128, sources=2, history=102400, tail=256,
              hot=4096, topk=2048, steps=32, warmup_steps=16, residency=None,
              capacity_frac=0.15, rho=0.9)
LONG = Config("long", 5, requests=32, sources=3, history=512000, tail=256,
              hot=8192, topk=2048, steps=16, residency=0.2, reuse_layers=3,
              shared_selection=True)

# host-copy profiling case: nothing optional-resident, so every selected row
# outside the tail is a hot-cache hit or a host fetch (1.2 GB pinned region,
# about 0.25 GB on the device)
MISS = Config("miss", 6, requests=16, sources=2, history=32768, tail=256, hot=4096,
              topk=2048, steps=16, residency=0.0)

# the same miss-heavy shape over a pinned region past the host link's
# translation reach: 32 requests x 2 sources x 768K-row histories (58 GB of
# pinned rows) with about 0.25 GB on the device; the host copy reads rows
# scattered over the whole region every step
WIDE = Config("wide", 7, requests=32, sources=2, history=786432, tail=256, hot=4096,
              topk=2048, steps=16, residency=0.0)

CONFIGS = {c.name: c for c in (TINY, C8, C64, C128, LONG, MISS, WIDE)}


class Workload:
    """All seeded inputs of one configuration.

    Step numbers are 1-based.  At step s every (request, source) first
    appends ``append[r, s-1]`` rows, then resolves its selection for the
    step over the new length ``length(r, s)``.
    """

    def __init__(self, cfg: Config, seed: int = SEED):
        self.cfg = cfg
        self.seed = seed
        c = cfg
        self.append = np.stack([
            append_counts(c.tag, r, c.total_steps, c.append_lo, c.append_hi, seed)
            for r in range(c.requests)]) if c.total_steps else \
            np.zeros((c.requests, 0), np.int32)
        # L after step s's append, s = 0..total_steps (s = 0: admission)
        self._len = np.concatenate(
            [np.full((c.requests, 1), c.history, np.int64),
             c.history + np.cumsum(self.append, axis=1, dtype=np.int64)], axis=1)
        self._sel = None

    # ---------------------------------------------------------- lengths
    def length(self, r: int, step: int) -> int:
        return int(self._len[r, step])

    # ---------------------------------------------------------- residency
    def resident_mask(self, r: int, s: int) -> np.ndarray:
        """uint8 per complete page: 1 = admitted optional-resident."""
        c = self.cfg
        if c.residency is None:  # admission-driven: admit everything first
            return np.ones(c.complete_pages, np.uint8)
        return residency(c.tag, s, r, c.complete_pages, c.resident_pages(),
                         self.seed)

    # ---------------------------------------------------------- payload
    def fill_host_rows(self, out_ptr: int, pair_stride_rows: int,
                       pairs=None, nthreads=None) -> None:
        """Imported rows [0, N) of each (r, s) pair (default: all pairs, in
        r-major order) into raw host memory with the given pair stride."""
        c = self.cfg
        if pairs is None:
            pairs = [(r, s) for r in range(c.requests) for s in range(c.sources)]
        payload_pairs_into(out_ptr, pair_stride_rows, c.tag,
                           [(s, r) for (r, s) in pairs], 0, c.history,
                           c.row_elems, self.seed, nthreads)

    def appended_rows(self, step: int, pairs=None) -> tuple[np.ndarray, np.ndarray]:
        """Rows appended at `step` for each (r, s) pair.

        Returns (counts [n_pairs], rows [n_pairs][append_hi][E] uint16);
        rows beyond a pair's count are zero.
        """
        c = self.cfg
        if pairs is None:
            pairs = [(r, s) for r in range(c.requests) for s in range(c.sources)]
        counts = np.array([self.append[r, step - 1] for (r, _) in pairs], np.int32)
        rows = np.zeros((len(pairs), c.append_hi, c.row_elems), np.uint16)
        for i, (r, s) in enumerate(pairs):
            n = int(counts[i])
            if n:
                p0 = self.length(r, step - 1)
                payload_pairs_into(rows[i].ctypes.data, n, c.tag, [(s, r)], p0,
                                   n, c.row_elems, self.seed, 1)
        return counts, rows

    # ---------------------------------------------------------- selections
    @property
    def sel_sources(self) -> int:
        return 1 if self.cfg.shared_selection else self.cfg.sources

    def _gen_pair(self, r: int, s: int, cdf, out) -> None:
        c = self.cfg
        perm = permutation(c.tag, s, r, c.history, self.seed)
        prev = None
        for step in range(1, c.total_steps + 1):
            L = self.length(r, step)
            if c.queries == 1:
                rows, z = select(c.tag, s, r, step, 0, L, c.history, c.topk,
                                 c.window, c.frac_recent, cdf, perm, prev,
                                 c.rho, None, self.seed)
                out[step - 1, r, s, 0] = rows
                prev = z
                continue
            core, _ = select(c.tag, s, r, step, 0, L, c.history, c.verify_core,
                             c.window, c.frac_recent, cdf, perm, None, 0.0,
                             None, self.seed)
            taken = core
            for q in range(c.queries):
                extra, _ = select(c.tag, s, r, step, q + 1, L, c.history,
                                  c.topk - c.verify_core, c.window,
                                  c.frac_recent, cdf, perm, None, 0.0, taken,
                                  self.seed)
                out[step - 1, r, s, q] = np.sort(np.concatenate([core, extra]))
                taken = np.concatenate([taken, extra])

    def selections(self, nthreads: int | None = None) -> np.ndarray:
        """int32 [total_steps][R][sel_sources][Q][k], generated once."""
        if self._sel is not None:
            return self._sel
        c = self.cfg
        out = np.empty((c.total_steps, c.requests, self.sel_sources, c.queries,
                        c.topk), np.int32)
        cdf = zipf_cdf(c.history, c.zipf_s)
        jobs = [(r, s) for r in range(c.requests) for s in range(self.sel_sources)]
        nthreads = nthreads or min(len(jobs), os.cpu_count() or 1)
        if nthreads <= 1:
            for r, s in jobs:
                self._gen_pair(r, s, cdf, out)
        else:
            with cf.ThreadPoolExecutor(nthreads) as ex:
                list(ex.map(lambda rs: self._gen_pair(rs[0], rs[1], cdf, out), jobs))
        self._sel = out
        return out

    def sel(self, step: int, r: int, s: int) -> np.ndarray:
        """[Q][k] selection of (r, s) at `step` (shared across sources when
        the configuration shares selections)."""
        return self.selections()[step - 1, r, 0 if self.cfg.shared_selection else s]


def drive_admission(api, cfg: Config, wl: Workload) -> None:
    """Admit every (request, source) in request order.

    Fixed-residency configurations admit each pair with its seeded resident
    page set.  Admission-driven ones (pool capacity a fraction of all pages)
    admit every pair resident-first; when an admission reports a deficit the
    caller reclaims whole earlier requests, oldest first, and admits again.

    `api` provides ``admit(r, s, mask) -> (rc, deficit)`` with rc 0 or
    'wouldwait', and ``reclaim(order, deficit) -> (rc, freed)``.
    """
    for r in range(cfg.requests):
        for s in range(cfg.sources):
            mask = wl.resident_mask(r, s)
            rc, deficit = api.admit(r, s, mask)
            if rc == 0:
                continue
            if rc != "wouldwait":
                raise RuntimeError(f"admit({r},{s}) failed: {rc}")
            rc2, freed = api.reclaim(list(range(r)), deficit)
            if rc2 != 0:
                raise RuntimeError(f"reclaim for ({r},{s}) failed: {rc2}")
            rc, deficit = api.admit(r, s, mask)
            if rc != 0:
                raise RuntimeError(f"admit({r},{s}) after reclaim failed: {rc}")

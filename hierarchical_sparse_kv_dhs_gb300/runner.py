"""Drive a synthetic workload through libdhs on one GPU.

Layout in HBM (all caller-owned, allocated once through torch):
  * the pool's four arenas (hot cache, tail ring, optional pages, metadata);
  * every step's selections, resident: int32 [steps][R][S_sel][Q][k];
  * every step's appended decode rows: [steps][R*S][a_max][row_bytes];
  * one location vector set uint32 [R][S][Q][k], one counter set
    uint32 [R][S][8] and one staging buffer [R][layers][Q][k][row_bytes],
    rewritten every step.
Pinned host memory: one registered buffer [R*S][max_rows][row_bytes] holding
every (request, source)'s imported rows, with room for the decode rows the
library writes through.

A decode step (``step``) is one ``dhs_decode_step``: every source's new
rows are appended, then R x layers items are resolved and gathered -- each
source's own resolution, then the gathers of all layers, Reuse layers
gathering source 0's location vector as DHS_ITEM_GATHER_ONLY items.  The
ctypes descriptors of every step are built before the first step, so a step
costs one C call.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from dhs_workload.configs import Config, Workload, drive_admission

from . import dhs


class _Admit:
    def __init__(self, run):
        self.run = run

    def admit(self, r, s, mask):
        rc, d = self.run.pool.admit(r, s, self.run.host_ptr(r, s), self.run.cfg.history, mask)
        return dhs.RC_NAMES[rc], d

    def reclaim(self, order, deficit):
        rc, f = self.run.pool.reclaim(order, deficit)
        return dhs.RC_NAMES[rc], f


def _align16(n: int) -> int:
    return (n + 15) // 16 * 16


def _field(block, offset: int, dtype, shape):
    """A typed view of bytes [offset, ...) of a uint8 block: of each row of a
    2-D block ([steps][bytes]), or of a 1-D block."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    if block.dim() == 2:
        return block[:, offset:offset + n].view(dtype).view(block.shape[0], *shape)
    return block[offset:offset + n].view(dtype).view(*shape)


class GpuRun:
    def __init__(self, cfg: Config, wl: Workload | None = None, device="cuda",
                 host_threads=None, gather_impl=None, payload_requests=None,
                 hugepages=True, union=False):
        """payload_requests: requests whose imported rows are generated
        (default all); the others' pinned rows stay zero -- for parity runs
        that compare sampled requests on workloads too large to fill.
        union: resolve in the union staging layout (DHS_ITEM_UNION): `loc`
        holds each source's union locations then DHS_END_LOC, `index` the
        entries' union ranks, and each layer's staging its first U rows."""
        self.cfg = c = cfg
        self.union = union
        self.wl = wl or Workload(cfg)
        self.device = torch.device(device)
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        torch.cuda.set_device(self.device)
        self.layers = [("resolve", s) for s in range(c.sources)] + \
            [("reuse", 0)] * c.reuse_layers
        self.pool = dhs.Pool(
            max_requests=c.requests, sources=c.sources, row_bytes=c.row_bytes,
            page_rows=c.page_rows, tail_rows=c.tail, hot_rows=c.hot,
            max_queries=c.queries, max_topk=c.topk, max_rows_per_request=c.max_rows,
            optional_pages=c.pool_pages(), device=self.device)
        if gather_impl is not None:
            self.pool.set_option(dhs.DHS_OPT_GATHER_IMPL, gather_impl)
        rb = c.row_bytes
        self.host = dhs.HostRows(c.pairs * c.max_rows * rb, hugepages=hugepages)
        pairs = None if payload_requests is None else [
            (r, s) for r in range(c.requests) for s in range(c.sources)
            if r in set(payload_requests)]
        if pairs is None:
            self.wl.fill_host_rows(self.host.ptr, c.max_rows, nthreads=host_threads)
        else:
            for (r, s) in pairs:  # pair (r, s) lives at its own offset
                self.wl.fill_host_rows(self.host_ptr(r, s), c.max_rows, [(r, s)],
                                       nthreads=host_threads)
        drive_admission(_Admit(self), c, self.wl)
        dhs.check(self.pool.flush(), "dhs_flush")

        dev = self.device
        Q, k = c.queries, c.topk
        sel = self.wl.selections()
        a_hi = c.append_hi
        # Each step's inputs lie in one block (selections, then appended rows)
        # and the step's outputs in another (locations, counters, union
        # indices), so that a caller with host buffers moves each with a
        # single copy.
        sel_b = _align16(sel[0].nbytes)
        rows_shape = (c.pairs, a_hi, c.row_elems)
        in_b = sel_b + _align16(int(np.prod(rows_shape)) * 2)
        self.step_in = torch.zeros((c.total_steps, in_b), dtype=torch.uint8, device=dev)
        self.sel = _field(self.step_in, 0, torch.int32, sel.shape[1:])
        self.sel.copy_(torch.from_numpy(sel))
        # appended rows of every step
        self.app_rows = _field(self.step_in, sel_b, torch.int16, rows_shape)
        loc_shape, cnt_shape = (c.requests, c.sources, Q, k), (c.requests, c.sources, 8)
        loc_b = _align16(int(np.prod(loc_shape)) * 4)
        cnt_b = _align16(int(np.prod(cnt_shape)) * 4)
        self.step_out = torch.zeros(loc_b + cnt_b + (loc_b if union else 0),
                                    dtype=torch.uint8, device=dev)
        self.loc = _field(self.step_out, 0, torch.int32, loc_shape)
        self.counters = _field(self.step_out, loc_b, torch.int32, cnt_shape)
        self.index = _field(self.step_out, loc_b + cnt_b, torch.int32, loc_shape) if union else None
        self.staging = torch.empty((c.requests, len(self.layers), Q, k, c.row_elems),
                                   dtype=torch.bfloat16, device=dev)
        pairs = [(r, s) for r in range(c.requests) for s in range(c.sources)]
        for step in range(1, c.total_steps + 1):
            _, rows = self.wl.appended_rows(step, pairs)
            self.app_rows[step - 1].copy_(torch.from_numpy(rows.view(np.int16)))
        self._build_descriptors()
        torch.cuda.synchronize(dev)

    def host_ptr(self, r, s):
        c = self.cfg
        return self.host.ptr + (r * c.sources + s) * c.max_rows * c.row_bytes

    def host_rows(self, r, s, row0, n):
        c = self.cfg
        base = (r * c.sources + s) * c.max_rows + row0
        a = self.host.array[base * c.row_bytes:(base + n) * c.row_bytes]
        return a.view(np.uint16).reshape(n, c.row_elems)

    # ---------------------------------------------------------- descriptors
    def _make_steps(self, loc, counters, index):
        """Step descriptors of every step with outputs in `loc`, `counters`
        (and union `index`): one dhs_step per step and one per layer."""
        c = self.cfg
        Q, k, rb = c.queries, c.topk, c.row_bytes
        steps, layer_steps = [], []
        loc0, cnt0 = loc.data_ptr(), counters.data_ptr()
        stg0 = self.staging.data_ptr()
        for step in range(1, c.total_steps + 1):
            items = []
            for r in range(c.requests):
                for layer, (kind, s) in enumerate(self.layers):
                    it = dhs.dhs_item()
                    it.req, it.src, it.queries, it.topk = r, s, Q, k
                    it.flags = dhs.DHS_ITEM_GATHER_ONLY if kind == "reuse" else 0
                    if self.union and kind != "reuse":
                        it.flags |= dhs.DHS_ITEM_UNION
                        it.index_dev = index[r, s].data_ptr()
                    ss = 0 if c.shared_selection else s
                    it.sel_dev = self.sel[step - 1, r, ss].data_ptr()
                    it.loc_dev = loc0 + ((r * c.sources + s) * Q * k) * 4
                    it.counters_dev = cnt0 + (r * c.sources + s) * 32
                    it.staging_dev = stg0 + ((r * len(self.layers) + layer) * Q * k) * rb
                    items.append(it)
            steps.append(dhs.make_step(step, items))
            nl = len(self.layers)
            layer_steps.append([dhs.make_step(step, items[l::nl]) for l in range(nl)])
        return steps, layer_steps

    def _build_descriptors(self):
        c = self.cfg
        self._steps, self._layer_steps = self._make_steps(self.loc, self.counters, self.index)
        self._outs = [(self.step_out, self._steps)]
        self._appends = []
        for step in range(1, c.total_steps + 1):
            apps = []
            for i, (r, s) in enumerate((r, s) for r in range(c.requests)
                                       for s in range(c.sources)):
                a = dhs.dhs_append_item()
                a.req, a.src = r, s
                a.count = int(self.wl.append[r, step - 1])
                a.rows_dev = self.app_rows[step - 1, i].data_ptr()
                apps.append(a)
            arr = (dhs.dhs_append_item * len(apps))(*apps)
            self._appends.append((arr, len(apps)))

    def output_block(self, i):
        """Output block `i` (locations, counters, union indices) laid out as
        step_out (block 0), with step descriptors that write it (host_io's
        `out_set`): a pipelined caller cycles through several blocks while
        earlier blocks' copies to the host are in flight."""
        while len(self._outs) <= i:
            blk = torch.zeros_like(self.step_out)
            off = lambda t: t.data_ptr() - self.step_out.data_ptr()
            view = lambda t: blk[off(t):off(t) + t.numel() * 4].view(torch.int32).view(t.shape)
            steps, _ = self._make_steps(view(self.loc), view(self.counters),
                                        view(self.index) if self.index is not None else None)
            self._outs.append((blk, steps))
        return self._outs[i][0]

    # ---------------------------------------------------------- stepping
    def append(self, step):
        arr, n = self._appends[step - 1]
        dhs.check(dhs.lib.dhs_append(self.pool.h, arr, n), "dhs_append")

    def resolve(self, step):
        st, _ = self._steps[step - 1]
        dhs.check(dhs.lib.dhs_resolve(self.pool.h, ctypes.byref(st)), "dhs_resolve")

    def gather(self, step):
        st, _ = self._steps[step - 1]
        dhs.check(dhs.lib.dhs_gather(self.pool.h, ctypes.byref(st)), "dhs_gather")

    def side_stream(self):
        if getattr(self, "_side", None) is None:
            self._side = torch.cuda.Stream(self.device)
        return self._side

    def prefetch(self, step):
        """Resolve every layer of the step on the side stream (dhs_prefetch)."""
        st, _ = self._steps[step - 1]
        dhs.check(dhs.lib.dhs_prefetch(self.pool.h, ctypes.byref(st),
                                       ctypes.c_void_p(self.side_stream().cuda_stream)),
                  "dhs_prefetch")

    def prefetch_layers(self, step, layers):
        """dhs_prefetch of the given layers' items (one step descriptor)."""
        key = (step, tuple(layers))
        cache = self.__dict__.setdefault("_pf_cache", {})
        if key not in cache:
            items = [it for l in layers for it in self._layer_steps[step - 1][l][1]
                     [: self._layer_steps[step - 1][l][0].n_items]]
            cache[key] = dhs.make_step(step, items)
        st, _ = cache[key]
        dhs.check(dhs.lib.dhs_prefetch(self.pool.h, ctypes.byref(st),
                                       ctypes.c_void_p(self.side_stream().cuda_stream)),
                  "dhs_prefetch")

    def resolve_layer(self, step, layer):
        st, _ = self._layer_steps[step - 1][layer]
        dhs.check(dhs.lib.dhs_resolve(self.pool.h, ctypes.byref(st)), "dhs_resolve")

    def gather_layer(self, step, layer, stream=None):
        """dhs_gather of one layer, or dhs_gather_on `stream` (torch stream)."""
        st, _ = self._layer_steps[step - 1][layer]
        if stream is None:
            dhs.check(dhs.lib.dhs_gather(self.pool.h, ctypes.byref(st)), "dhs_gather")
        else:
            dhs.check(dhs.lib.dhs_gather_on(self.pool.h, ctypes.byref(st),
                                            ctypes.c_void_p(stream.cuda_stream)),
                      "dhs_gather_on")

    def step(self, step, fused=True):
        """One decode step: append, then resolve + gather every layer -- one
        dhs_decode_step call (fused=True), dhs_append, dhs_resolve and
        dhs_gather (False), or dhs_append, dhs_prefetch on a side stream and
        dhs_gather ("prefetch")."""
        if fused == "prefetch":
            self.append(step)
            self.prefetch(step)
            self.gather(step)
            return
        if not fused:
            self.append(step)
            self.resolve(step)
            self.gather(step)
            return
        arr, n = self._appends[step - 1]
        st, _ = self._steps[step - 1]
        dhs.check(dhs.lib.dhs_decode_step(self.pool.h, arr, n, ctypes.byref(st)),
                  "dhs_decode_step")

    def host_io(self, step, ins, outs, out_set=0):
        """Prebuilt arguments of dhs_decode_step_host for `step`: `ins` /
        `outs` are lists of (dst, src, bytes) host<->device copies; the step
        writes output block `out_set` (output_block)."""
        arr, n = self._appends[step - 1]
        self.output_block(out_set)
        st, _ = self._outs[out_set][1][step - 1]
        cin = (dhs.dhs_copy * max(1, len(ins)))(*[dhs.dhs_copy(*c) for c in ins])
        cout = (dhs.dhs_copy * max(1, len(outs)))(*[dhs.dhs_copy(*c) for c in outs])
        return (self.pool.h, cin, len(ins), arr, n, ctypes.byref(st), cout, len(outs))

    def step_host(self, step, ins=None, outs=None, io=None, wait=True, in_stream=None,
                  out_stream=None):
        """dhs_decode_step_host with prebuilt `io` (host_io) or with ins/outs;
        returns after the outputs have landed in host memory, or (wait=False,
        dhs_decode_step_host_async) once everything is enqueued, the copies on
        `in_stream` / `out_stream` (torch streams; None = the pool's)."""
        io = io or self.host_io(step, ins, outs)
        if wait:
            dhs.check(dhs.lib.dhs_decode_step_host(*io), "dhs_decode_step_host")
            return
        h, cin, nin, arr, n, st, cout, nout = io
        sin = ctypes.c_void_p(in_stream.cuda_stream if in_stream is not None else None)
        sout = ctypes.c_void_p(out_stream.cuda_stream if out_stream is not None else None)
        dhs.check(dhs.lib.dhs_decode_step_host_async(h, cin, nin, sin, arr, n, st, cout, nout,
                                                     sout), "dhs_decode_step_host_async")

    def reset(self):
        """Release every request and admit it again: the pool returns to its
        state before step 1 (stream-ordered; no synchronisation)."""
        for r in range(self.cfg.requests):
            dhs.check(self.pool.release(r), "dhs_release")
        drive_admission(_Admit(self), self.cfg, self.wl)
        dhs.check(self.pool.flush(), "dhs_flush")

    def status(self):
        return self.pool.status()

    def close(self):
        self.pool.close()
        self.host.close()


class LoadStepGpu:
    """The load-step schedule (dhs_workload.loadstep.run) over the C ABI with
    every step as one batched dhs_decode_step, timed with CUDA events on the
    pool's stream: decode steps, device admissions, deferred backups and
    refills (whose host-to-device copies are enqueued by the dhs_flush the
    refill is followed by)."""

    def __init__(self, max_topk: int, device="cuda"):
        self.k = max_topk
        self.device = torch.device(device)
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        torch.cuda.set_device(self.device)
        self.times = {"step": [], "admit": [], "backup": [], "refill": []}
        self.bytes = {"admit": 0, "backup": 0, "refill": 0}

    def _timed(self, kind, fn, nbytes=0):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        out = fn()
        e1.record()
        e1.synchronize()
        self.times[kind].append(e0.elapsed_time(e1) / 1e3)
        if kind in self.bytes:
            self.bytes[kind] += nbytes
        return out

    def new_pool(self, R, S, T, B, E, PR, max_rows, cap, reserve):
        self.R, self.S, self.E, self.PR = R, S, E, PR
        self.rb = E * 2
        self.max_rows = max_rows
        self.pool = dhs.Pool(max_requests=R, sources=S, row_bytes=self.rb, page_rows=PR,
                             tail_rows=T, hot_rows=B, max_queries=1, max_topk=self.k,
                             max_rows_per_request=max_rows, optional_pages=cap,
                             admission_reserve_pages=reserve, device=self.device)
        self.host = dhs.HostRows(R * S * max_rows * self.rb, hugepages=False)
        dev = self.device
        self.sel = torch.zeros((R * S, self.k), dtype=torch.int32, device=dev)
        self.loc = torch.zeros((R * S, self.k), dtype=torch.int32, device=dev)
        self.cnt = torch.zeros((R * S, 8), dtype=torch.int32, device=dev)
        self.stg = torch.empty((R * S, self.k, E), dtype=torch.int16, device=dev)
        self.app = torch.zeros((R * S, E), dtype=torch.int16, device=dev)

    def _host_ptr(self, r, s):
        return self.host.ptr + (r * self.S + s) * self.max_rows * self.rb

    def admit_device(self, r, s, N, mask, rows):
        dev = torch.from_numpy(np.ascontiguousarray(rows).view(np.int16)).to(self.device)
        torch.cuda.synchronize(self.device)
        rc, d = self._timed("admit", lambda: self.pool.admit_device(
            r, s, dev.data_ptr(), self._host_ptr(r, s), N, mask), N * self.rb)
        return dhs.RC_NAMES[rc], d

    def release(self, r):
        return dhs.RC_NAMES[self.pool.release(r)]

    def reclaim(self, order, deficit):
        rc, f = self.pool.reclaim(order, deficit)
        return dhs.RC_NAMES[rc], f

    def refill(self, n):
        rc, k = self.pool.refill(n)
        if k:
            self._timed("refill", lambda: dhs.check(self.pool.flush(), "dhs_flush"),
                        k * self.PR * self.rb)
        return dhs.RC_NAMES[rc], k

    def backup(self, n):
        rc, k = self._timed("backup", lambda: self.pool.backup(n))
        if k:
            self.bytes["backup"] += k * self.PR * self.rb
        else:
            self.times["backup"].pop()
        return dhs.RC_NAMES[rc], k

    def used(self):
        return self.pool.used()

    def pending_backup(self):
        return self.pool.pending_backup()

    def decode_step(self, step, work):
        apps, items = [], []
        for i, (r, s, row, sel) in enumerate(work):
            p = r * self.S + s
            self.app[p].copy_(torch.from_numpy(np.ascontiguousarray(row[0]).view(np.int16)))
            self.sel[p].copy_(torch.from_numpy(np.ascontiguousarray(sel, np.int32)))
            a = dhs.dhs_append_item()
            a.req, a.src, a.count, a.rows_dev = r, s, 1, self.app[p].data_ptr()
            apps.append(a)
            it = dhs.dhs_item()
            it.req, it.src, it.queries, it.topk = r, s, 1, len(sel)
            it.sel_dev, it.loc_dev = self.sel[p].data_ptr(), self.loc[p].data_ptr()
            it.counters_dev, it.staging_dev = self.cnt[p].data_ptr(), self.stg[p].data_ptr()
            items.append(it)
        arr = (dhs.dhs_append_item * len(apps))(*apps)
        st, keep = dhs.make_step(step, items)
        torch.cuda.synchronize(self.device)
        self._timed("step", lambda: dhs.check(
            dhs.lib.dhs_decode_step(self.pool.h, arr, len(apps), ctypes.byref(st)),
            "dhs_decode_step"))
        rc, flags = self.pool.status()
        if rc != 0:
            raise RuntimeError(f"device status {rc} flags {flags}")
        cnt = self.cnt.cpu().numpy().view(np.uint32)
        loc = self.loc.cpu().numpy().view(np.uint32)
        return [(0, loc[r * self.S + s, : len(sel)], cnt[r * self.S + s])
                for (r, s, _, sel) in work]

    def close(self):
        torch.cuda.synchronize(self.device)
        self.pool.close()
        self.host.close()

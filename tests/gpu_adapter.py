"""Adapter that drives the CUDA library (through its C ABI) with the same
calls as the oracle adapter, for the golden traces and small parity runs."""
from __future__ import annotations

import numpy as np
import torch

from hierarchical_sparse_kv_dhs_gb300 import dhs


class GpuAdapter:
    def __init__(self, max_queries=4, max_topk=16):
        self.mq, self.mk = max_queries, max_topk

    def new_pool(self, R, S, T, B, E, PR, max_rows, cap, reserve):
        self.R, self.S, self.T, self.B, self.E, self.PR = R, S, T, B, E, PR
        self.max_rows = max_rows
        self.rb = E * 2
        self.pool = dhs.Pool(max_requests=R, sources=S, row_bytes=self.rb, page_rows=PR,
                             tail_rows=T, hot_rows=B, max_queries=self.mq,
                             max_topk=self.mk, max_rows_per_request=max_rows,
                             optional_pages=cap, admission_reserve_pages=reserve)
        self.host = dhs.HostRows(R * S * max_rows * self.rb)
        self.lengths = {}

    def _host_off(self, r, s):
        return (r * self.S + s) * self.max_rows * self.rb

    def admit(self, r, s, N, mask, host):
        off = self._host_off(r, s)
        self.host.array[off: off + N * self.rb] = np.ascontiguousarray(host).view(np.uint8).ravel()
        rc, d = self.pool.admit(r, s, self.host.ptr + off, N, mask)
        if rc == 0:
            self.lengths[(r, s)] = N
        return dhs.RC_NAMES[rc], d

    def admit_device(self, r, s, N, mask, rows):
        off = self._host_off(r, s)
        # the host copy starts empty: only this call's copies and later
        # backups may fill it
        self.host.array[off: off + self.max_rows * self.rb] = 0
        dev = torch.from_numpy(np.ascontiguousarray(rows).view(np.int16).copy()).cuda()
        rc, d = self.pool.admit_device(r, s, dev.data_ptr(), self.host.ptr + off, N, mask)
        torch.cuda.synchronize()  # dev is read by the copies just enqueued
        if rc == 0:
            self.lengths[(r, s)] = N
        return dhs.RC_NAMES[rc], d

    def admit_window(self, r, s, N, rows):
        m = min(N, self.T)
        dev = torch.from_numpy(np.ascontiguousarray(rows[:m]).view(np.int16).copy()).cuda()
        rc = self.pool.admit_window(r, s, dev.data_ptr() if m else None, N)
        torch.cuda.synchronize()  # dev is read by the copies just enqueued
        if rc == 0:
            self.lengths[(r, s)] = N
        return dhs.RC_NAMES[rc]

    def backup(self, n):
        rc, k = self.pool.backup(n)
        torch.cuda.synchronize()
        return dhs.RC_NAMES[rc], k

    def refill(self, n):
        rc, k = self.pool.refill(n)
        return dhs.RC_NAMES[rc], k

    def pending_backup(self):
        return self.pool.pending_backup()

    def host_rows(self, r, s, row0, n):
        torch.cuda.synchronize()
        off = self._host_off(r, s) + row0 * self.rb
        return self.host.array[off: off + n * self.rb].view(np.uint16).reshape(n, self.E).copy()

    def reclaim(self, order, deficit):
        rc, f = self.pool.reclaim(order, deficit)
        torch.cuda.synchronize()
        return dhs.RC_NAMES[rc], f

    def release(self, r):
        return dhs.RC_NAMES[self.pool.release(r)]

    def used(self):
        return self.pool.used()

    def pages(self, r, s):
        return self.pool.read_state(r, s)[2]

    def append(self, r, s, count, rows):
        dev = torch.from_numpy(np.ascontiguousarray(rows).view(np.int16).copy()).cuda()
        it = dhs.dhs_append_item()
        it.req, it.src, it.count, it.rows_dev = r, s, count, dev.data_ptr()
        rc = dhs.dhs_append(self.pool.h, [it])
        torch.cuda.synchronize()
        return dhs.RC_NAMES[rc]

    def resolve(self, step, r, s, sel):
        sel = np.ascontiguousarray(sel, np.int32)
        Q, k = sel.shape
        d_sel = torch.from_numpy(sel).cuda()
        d_loc = torch.zeros(max(Q * k, 1), dtype=torch.int32, device="cuda")
        d_cnt = torch.full((8,), -7, dtype=torch.int32, device="cuda")
        it = dhs.dhs_item()
        it.req, it.src, it.queries, it.topk = r, s, Q, k
        it.sel_dev, it.loc_dev, it.counters_dev = d_sel.data_ptr(), d_loc.data_ptr(), d_cnt.data_ptr()
        st, keep = dhs.make_step(step, [it])
        dhs.check(dhs.dhs_resolve(self.pool.h, st), "dhs_resolve")
        torch.cuda.synchronize()
        info = self.pool.read_state(r, s)[3]
        code = int(info[3])
        rc_status, flags = self.pool.status()
        want_flag = {0: 0, dhs.DHS_ERANGE: dhs.DHS_STATUS_ERANGE,
                     dhs.DHS_EBUDGET: dhs.DHS_STATUS_EBUDGET}[code]
        assert flags == want_flag, (code, flags)
        loc = d_loc[: Q * k].cpu().numpy().view(np.uint32).reshape(Q, k)
        cnt = d_cnt.cpu().numpy().view(np.uint32)
        return dhs.RC_NAMES[code], loc, cnt

    def gather(self, loc):
        loc = np.ascontiguousarray(loc, np.uint32).ravel()
        d_loc = torch.from_numpy(loc.view(np.int32).copy()).cuda()
        d_stg = torch.full((loc.size, self.E), 0x5555, dtype=torch.int16, device="cuda")
        it = dhs.dhs_item()
        it.queries, it.topk = 1, loc.size
        it.flags = dhs.DHS_ITEM_GATHER_ONLY
        it.loc_dev, it.staging_dev = d_loc.data_ptr(), d_stg.data_ptr()
        st, keep = dhs.make_step(1, [it])
        dhs.check(dhs.dhs_gather(self.pool.h, st), "dhs_gather")
        torch.cuda.synchronize()
        rc, flags = self.pool.status()
        assert rc == 0 and flags == 0
        return d_stg.cpu().numpy().view(np.uint16)

    def state(self, r, s):
        tags, stamps, _, _ = self.pool.read_state(r, s)
        return tags, stamps

"""CPU oracle of the hierarchical sparse KV resolve + gather path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product library
never imports, links or runs anything here.  The arithmetic is in
``dhs_oracle.c`` (plain C, compiled with gcc); this module wraps it with
ctypes and adds a whole-workload driver.

Every function of ``dhs_oracle.c`` is pinned by the CPU tests (hand-worked
fixtures under tests/golden, closed forms, a stack-distance LRU identity,
brute force on tiny inputs, byte truth against the payload generator).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# DHS_ORACLE_SRC names another copy of dhs_oracle.c to build and load instead
# (the mutation harness in tests/ plants one mistake per copy); its library
# is built beside it.
_SRC = os.environ.get("DHS_ORACLE_SRC") or os.path.join(_HERE, "dhs_oracle.c")
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(_SRC)), "liborc.so")
_lib = None
_lock = threading.Lock()

NO_LOC = 0xFFFFFFFF
END_LOC = 0xFFFFFFFE  # past the end of a union location list
TIER_TAIL, TIER_OPT, TIER_HOT = 0, 1, 2
RC_NAMES = {0: 0, -1: "einval", -2: "enomem", -3: "wouldwait", -4: "ebudget",
            -5: "erange", -8: "estate"}
COUNTERS = ("entries", "unique", "tail", "opt", "hot", "host", "scan_max",
            "evicted")


def source_path() -> str:
    """The oracle source this module builds and loads."""
    return _SRC


def build(force: bool = False) -> str:
    """Compile dhs_oracle.c into liborc.so (gcc, -O2, no CUDA)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared",
                           "-o", tmp, _SRC])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def declare(L: ctypes.CDLL) -> ctypes.CDLL:
    """Set the argument and result types of the oracle's entry points on a
    loaded copy of the library."""
    i32, i64, u32, vp = (ctypes.c_int32, ctypes.c_int64,
                         ctypes.c_uint32, ctypes.c_void_p)
    L.orc_pool_new.restype = vp
    L.orc_pool_new.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, i64]
    L.orc_pool_free.restype = None
    L.orc_pool_free.argtypes = [vp]
    L.orc_pool_used.restype = i64
    L.orc_pool_used.argtypes = [vp]
    L.orc_admit.restype = ctypes.c_int
    L.orc_admit.argtypes = [vp, i32, i32, vp, i64, vp, vp]
    L.orc_reclaim.restype = ctypes.c_int
    L.orc_reclaim.argtypes = [vp, vp, i32, i64, vp]
    L.orc_release.restype = ctypes.c_int
    L.orc_release.argtypes = [vp, i32]
    L.orc_append.restype = ctypes.c_int
    L.orc_append.argtypes = [vp, i32, i32, i32, vp]
    L.orc_resolve.restype = ctypes.c_int
    L.orc_resolve.argtypes = [vp, u32, i32, i32, i32, i32, vp, vp, vp]
    L.orc_admit_device.restype = ctypes.c_int
    L.orc_admit_device.argtypes = [vp, i32, i32, vp, i64, vp, vp]
    L.orc_backup.restype = ctypes.c_int
    L.orc_backup.argtypes = [vp, i64, vp]
    L.orc_refill.restype = ctypes.c_int
    L.orc_refill.argtypes = [vp, i64, vp]
    L.orc_pending_backup.restype = i64
    L.orc_pending_backup.argtypes = [vp]
    L.orc_resolve_union.restype = ctypes.c_int
    L.orc_resolve_union.argtypes = [vp, u32, i32, i32, i32, i32, vp, vp, vp, vp]
    L.orc_gather.restype = ctypes.c_int
    L.orc_gather.argtypes = [vp, vp, i64, vp]
    L.orc_read_state.restype = ctypes.c_int
    L.orc_read_state.argtypes = [vp, i32, i32, vp, vp, vp, vp]
    L.orc_read_rows.restype = ctypes.c_int
    L.orc_read_rows.argtypes = [vp, i32, i32, ctypes.c_int, i64, i64, vp]
    L.orc_check.restype = ctypes.c_int
    L.orc_check.argtypes = [vp, i32, i32]
    L.orc_admit_window.restype = ctypes.c_int
    L.orc_admit_window.argtypes = [vp, i32, i32, vp, i64]
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return a.ctypes.data


class OraclePool:
    """One oracle pool: R requests x S sources, tail T, hot cache B rows of
    E bf16 elements, pages of PR rows, optional capacity in pages."""

    def __init__(self, R, S, T, B, E, PR, max_rows, capacity, reserve=0):
        self.R, self.S, self.T, self.B, self.E, self.PR = R, S, T, B, E, PR
        self.max_rows = max_rows
        self.pages_max = -(-max_rows // PR)
        self._h = lib().orc_pool_new(R, S, T, B, E, PR, max_rows, capacity, reserve)
        if not self._h:
            raise ValueError("orc_pool_new rejected the configuration")

    def close(self):
        if self._h:
            lib().orc_pool_free(self._h)
            self._h = None

    __del__ = close

    def used(self) -> int:
        return lib().orc_pool_used(self._h)

    def admit(self, r, s, N, mask=None, host_rows=None):
        d = ctypes.c_int64(0)
        if mask is not None:
            mask = np.ascontiguousarray(mask, dtype=np.uint8)
        if host_rows is not None:
            host_rows = np.ascontiguousarray(host_rows, dtype=np.uint16)
            assert host_rows.size >= N * self.E
        rc = lib().orc_admit(self._h, r, s, _p(host_rows), N, _p(mask),
                             ctypes.byref(d))
        return RC_NAMES[rc], d.value

    def admit_device(self, r, s, N, mask=None, rows=None):
        """Resident-first admission of rows held on the device (backup of the
        resident pages deferred)."""
        d = ctypes.c_int64(0)
        if mask is not None:
            mask = np.ascontiguousarray(mask, dtype=np.uint8)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.uint16)
            assert rows.size >= N * self.E
        rc = lib().orc_admit_device(self._h, r, s, _p(rows), N, _p(mask), ctypes.byref(d))
        return RC_NAMES[rc], d.value

    def admit_window(self, r, s, N, rows=None):
        """Admit a window source: the tail ring is its only storage; `rows`
        are the window's rows [N - min(N, T), N)."""
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.uint16)
            assert rows.size >= min(N, self.T) * self.E
        return RC_NAMES[lib().orc_admit_window(self._h, r, s, _p(rows), N)]

    def backup(self, max_pages):
        n = ctypes.c_int64(0)
        rc = lib().orc_backup(self._h, max_pages, ctypes.byref(n))
        return RC_NAMES[rc], n.value

    def refill(self, max_pages):
        n = ctypes.c_int64(0)
        rc = lib().orc_refill(self._h, max_pages, ctypes.byref(n))
        return RC_NAMES[rc], n.value

    def pending_backup(self):
        return int(lib().orc_pending_backup(self._h))

    def reclaim(self, order, deficit):
        o = np.ascontiguousarray(order, dtype=np.int32)
        f = ctypes.c_int64(0)
        rc = lib().orc_reclaim(self._h, _p(o) if len(o) else None, len(o),
                               deficit, ctypes.byref(f))
        return RC_NAMES[rc], f.value

    def release(self, r):
        return RC_NAMES[lib().orc_release(self._h, r)]

    def append(self, r, s, count, rows=None):
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.uint16)
        return RC_NAMES[lib().orc_append(self._h, r, s, count, _p(rows))]

    def resolve(self, step, r, s, sel):
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        if sel.ndim == 1:
            sel = sel[None]
        Q, k = sel.shape
        loc = np.empty(max(Q * k, 1), np.uint32)
        cnt = np.empty(8, np.uint32)
        rc = lib().orc_resolve(self._h, step, r, s, Q, k, _p(sel), _p(loc), _p(cnt))
        return RC_NAMES[rc], loc[: Q * k].reshape(Q, k), cnt

    def resolve_union(self, step, r, s, sel):
        """Union staging layout: (rc, loc [Q*k] -- U union locations then
        END_LOC, index [Q][k] into the union, counters)."""
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        if sel.ndim == 1:
            sel = sel[None]
        Q, k = sel.shape
        loc = np.empty(max(Q * k, 1), np.uint32)
        idx = np.empty(max(Q * k, 1), np.int32)
        cnt = np.empty(8, np.uint32)
        rc = lib().orc_resolve_union(self._h, step, r, s, Q, k, _p(sel), _p(loc),
                                     _p(idx), _p(cnt))
        return RC_NAMES[rc], loc[: Q * k], idx[: Q * k].reshape(Q, k), cnt

    def gather(self, loc):
        loc = np.ascontiguousarray(loc, dtype=np.uint32)
        out = np.empty(loc.shape + (self.E,), np.uint16)
        rc = lib().orc_gather(self._h, _p(loc.ravel()), loc.size, _p(out))
        return RC_NAMES[rc], out

    def state(self, r, s):
        tags = np.empty(self.B, np.int32)
        stamps = np.empty(self.B, np.uint32)
        ps = np.empty(self.pages_max, np.int32)
        ln = np.empty(3, np.int64)
        rc = lib().orc_read_state(self._h, r, s, _p(tags), _p(stamps), _p(ps), _p(ln))
        assert rc == 0
        return tags, stamps, ps, (int(ln[0]), int(ln[1]), int(ln[2]))

    def rows(self, r, s, which, row0, n):
        out = np.empty((n, self.E), np.uint16)
        rc = lib().orc_read_rows(self._h, r, s, which, row0, n, _p(out))
        if rc != 0:
            raise ValueError(f"orc_read_rows: {RC_NAMES[rc]}")
        return out

    def check(self, r, s) -> int:
        return lib().orc_check(self._h, r, s)


def decode(loc: np.ndarray):
    """(tier, index) arrays of a location vector."""
    loc = np.asarray(loc, np.uint32)
    return loc >> 30, loc & 0x3FFFFFFF

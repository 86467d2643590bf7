"""ctypes binding of libdhs (include/dhs.h): same names, argument marshalling
only.  Every step of the resolve + gather path runs in the library's CUDA
kernels; nothing here computes a location, a victim or a byte.

PyTorch supplies device memory and streams; pinned host rows come from
``HostRows`` (page-aligned anonymous memory registered as mapped pinned
memory with the CUDA runtime).

Importing this module fails loudly when libdhs.so has not been built.
"""
from __future__ import annotations

import ctypes
import mmap
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdhs.so")

DHS_OK = 0
DHS_EINVAL = -1
DHS_ENOMEM = -2
DHS_EWOULDWAIT = -3
DHS_EBUDGET = -4
DHS_ERANGE = -5
DHS_ETIMEDOUT = -6
DHS_ECUDA = -7
DHS_ESTATE = -8
RC_NAMES = {0: 0, -1: "einval", -2: "enomem", -3: "wouldwait", -4: "ebudget",
            -5: "erange", -6: "etimedout", -7: "ecuda", -8: "estate"}

DHS_TIER_TAIL, DHS_TIER_OPT, DHS_TIER_HOT = 0, 1, 2
DHS_NO_LOC = 0xFFFFFFFF
DHS_END_LOC = 0xFFFFFFFE
DHS_NUM_COUNTERS = 8
DHS_STATUS_ERANGE, DHS_STATUS_EBUDGET, DHS_STATUS_ELOC, DHS_STATUS_ETIMEDOUT = 1, 2, 4, 8
DHS_ITEM_GATHER_ONLY = 1
DHS_ITEM_UNION = 2
DHS_OPT_COPY_CTAS = 1
DHS_OPT_GATHER_IMPL = 2
DHS_OPT_TRACE = 3
DHS_OPT_EARLY = 4
DHS_OPT_FRESH_LIST = 5
DHS_OPT_GATHER_TPC = 6
DHS_OPT_STAGE_MISSES = 7
DHS_OPT_MARK_POLLS = 8
DHS_OPT_COPY_PDL = 9
DHS_OPT_RESOLVE_PAIRED = 10
DHS_OPT_COPY_STEAL = 11
DHS_OPT_RESOLVE_CTAS = 12
DHS_BUF_HOT, DHS_BUF_TAIL, DHS_BUF_OPT, DHS_BUF_META = range(4)

_i32, _i64, _u32, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p


class dhs_pool_config(ctypes.Structure):
    _fields_ = [("max_requests", _i32), ("sources", _i32), ("row_bytes", _i32),
                ("page_rows", _i32), ("tail_rows", _i32), ("hot_rows", _i32),
                ("max_queries", _i32), ("max_topk", _i32),
                ("max_rows_per_request", _i64), ("optional_pages", _i64),
                ("admission_reserve_pages", _i64),
                ("hot_dev", _vp), ("tail_dev", _vp), ("opt_dev", _vp),
                ("meta_dev", _vp), ("stream", _vp)]


class dhs_append_item(ctypes.Structure):
    _fields_ = [("req", _i32), ("src", _i32), ("count", _i32), ("reserved", _i32),
                ("rows_dev", _vp)]


class dhs_item(ctypes.Structure):
    _fields_ = [("req", _i32), ("src", _i32), ("queries", _i32), ("topk", _i32),
                ("flags", _u32), ("reserved", _i32), ("sel_dev", _vp),
                ("loc_dev", _vp), ("staging_dev", _vp), ("counters_dev", _vp),
                ("index_dev", _vp)]


class dhs_copy(ctypes.Structure):
    _fields_ = [("dst", _vp), ("src", _vp), ("bytes", ctypes.c_size_t)]


class dhs_step(ctypes.Structure):
    _fields_ = [("step", _u32), ("n_items", _i32), ("items", ctypes.POINTER(dhs_item))]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run hierarchical_sparse_kv_dhs_gb300.build.build() "
            "(nvcc, sm_103a) first -- there is no fallback path")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "dhs_pool_bytes": (ctypes.c_int, [P(dhs_pool_config), P(ctypes.c_size_t)]),
        "dhs_pool_create": (ctypes.c_int, [P(dhs_pool_config), P(_vp)]),
        "dhs_pool_destroy": (None, [_vp]),
        "dhs_admit": (ctypes.c_int, [_vp, _i32, _i32, _vp, _i64, _vp, P(_i64)]),
        "dhs_reclaim": (ctypes.c_int, [_vp, _vp, _i32, _i64, P(_i64)]),
        "dhs_release": (ctypes.c_int, [_vp, _i32]),
        "dhs_prefetch": (ctypes.c_int, [_vp, _vp, _vp]),
        "dhs_gather_on": (ctypes.c_int, [_vp, _vp, _vp]),
        "dhs_decode_step_host": (ctypes.c_int, [_vp, _vp, _i32, _vp, _i32, _vp, _vp, _i32]),
        "dhs_decode_step_host_async": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, _i32, _vp,
                                                      _vp, _i32, _vp]),
        "dhs_admit_device": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _i64, _vp, P(_i64)]),
        "dhs_admit_window": (ctypes.c_int, [_vp, _i32, _i32, _vp, _i64]),
        "dhs_backup": (ctypes.c_int, [_vp, _i64, P(_i64)]),
        "dhs_pending_backup": (_i64, [_vp]),
        "dhs_refill": (ctypes.c_int, [_vp, _i64, P(_i64)]),
        "dhs_pool_used": (_i64, [_vp]),
        "dhs_flush": (ctypes.c_int, [_vp]),
        "dhs_append": (ctypes.c_int, [_vp, P(dhs_append_item), _i32]),
        "dhs_resolve": (ctypes.c_int, [_vp, P(dhs_step)]),
        "dhs_gather": (ctypes.c_int, [_vp, P(dhs_step)]),
        "dhs_resolve_gather": (ctypes.c_int, [_vp, P(dhs_step)]),
        "dhs_decode_step": (ctypes.c_int, [_vp, P(dhs_append_item), _i32, P(dhs_step)]),
        "dhs_status": (ctypes.c_int, [_vp, P(_u32)]),
        "dhs_read_state": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _vp]),
        "dhs_set_option": (ctypes.c_int, [_vp, _i32, _i64]),
        "dhs_get_option": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(_i64)]),
        "dhs_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


class DhsError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {lib.dhs_strerror(code).decode()} ({code})")


def check(code, what=""):
    if code != DHS_OK:
        raise DhsError(code, what)
    return code


# ------------------------------------------------------------ C-named calls

def dhs_pool_bytes(cfg: dhs_pool_config) -> list[int]:
    out = (ctypes.c_size_t * 4)()
    check(lib.dhs_pool_bytes(ctypes.byref(cfg), out), "dhs_pool_bytes")
    return list(out)


def dhs_pool_create(cfg: dhs_pool_config) -> int:
    h = _vp()
    check(lib.dhs_pool_create(ctypes.byref(cfg), ctypes.byref(h)), "dhs_pool_create")
    return h.value


def dhs_pool_destroy(h: int) -> None:
    lib.dhs_pool_destroy(h)


def dhs_admit(h, req, src, host_ptr, n_rows, mask=None):
    d = _i64(0)
    m = None
    if mask is not None:
        mask = np.ascontiguousarray(mask, np.uint8)
        m = mask.ctypes.data
    rc = lib.dhs_admit(h, req, src, host_ptr, n_rows, m, ctypes.byref(d))
    return rc, d.value


def dhs_reclaim(h, order, deficit):
    o = np.ascontiguousarray(order, np.int32)
    f = _i64(0)
    rc = lib.dhs_reclaim(h, o.ctypes.data if len(o) else None, len(o), deficit,
                         ctypes.byref(f))
    return rc, f.value


def dhs_release(h, req):
    return lib.dhs_release(h, req)


def dhs_admit_device(h, req, src, dev_ptr, host_ptr, n_rows, mask=None):
    d = _i64(0)
    m = None
    if mask is not None:
        mask = np.ascontiguousarray(mask, np.uint8)
        m = mask.ctypes.data
    rc = lib.dhs_admit_device(h, req, src, dev_ptr, host_ptr, n_rows, m, ctypes.byref(d))
    return rc, d.value


def dhs_admit_window(h, req, src, dev_ptr, n_rows):
    return lib.dhs_admit_window(h, req, src, dev_ptr, n_rows)


def dhs_backup(h, max_pages):
    n = _i64(0)
    rc = lib.dhs_backup(h, max_pages, ctypes.byref(n))
    return rc, n.value


def dhs_refill(h, max_pages):
    n = _i64(0)
    rc = lib.dhs_refill(h, max_pages, ctypes.byref(n))
    return rc, n.value


def dhs_pool_used(h):
    return lib.dhs_pool_used(h)


def dhs_flush(h):
    return lib.dhs_flush(h)


def dhs_append(h, items):
    arr = (dhs_append_item * max(1, len(items)))(*items)
    return lib.dhs_append(h, arr, len(items))


def make_step(step: int, items) -> tuple:
    """A dhs_step plus the item array that must stay alive with it."""
    arr = (dhs_item * max(1, len(items)))(*items)
    return dhs_step(step, len(items), arr), arr


def dhs_resolve(h, st: dhs_step):
    return lib.dhs_resolve(h, ctypes.byref(st))


def dhs_gather(h, st: dhs_step):
    return lib.dhs_gather(h, ctypes.byref(st))


def dhs_resolve_gather(h, st: dhs_step):
    return lib.dhs_resolve_gather(h, ctypes.byref(st))


def dhs_decode_step(h, appends, st: dhs_step):
    arr = (dhs_append_item * max(1, len(appends)))(*appends)
    return lib.dhs_decode_step(h, arr, len(appends), ctypes.byref(st))


def dhs_status(h):
    f = _u32(0)
    rc = lib.dhs_status(h, ctypes.byref(f))
    return rc, f.value


def dhs_set_option(h, key, value):
    return lib.dhs_set_option(h, key, value)


def dhs_get_option(h, key):
    v = _i64(0)
    rc = lib.dhs_get_option(h, key, ctypes.byref(v))
    return rc, v.value


def dhs_read_state(h, req, src, B, pages_max):
    tags = np.empty(B, np.int32)
    stamps = np.empty(B, np.uint32)
    pages = np.empty(pages_max, np.int32)
    info = np.empty(4, np.int64)
    check(lib.dhs_read_state(h, req, src, tags.ctypes.data, stamps.ctypes.data,
                             pages.ctypes.data, info.ctypes.data), "dhs_read_state")
    return tags, stamps, pages, info


# ------------------------------------------------------------ host memory

class HostRows:
    """Page-aligned host memory registered as mapped pinned memory.

    ``array`` is a uint8 numpy view; ``ptr`` is the host address the library
    receives (it derives the device-visible address itself).
    """

    def __init__(self, nbytes: int, hugepages: bool = True):
        import torch
        self.nbytes = max(int(nbytes), 4096)
        self._mm = mmap.mmap(-1, self.nbytes)
        if hugepages and hasattr(mmap, "MADV_HUGEPAGE"):
            # ask for transparent huge pages (the GPU reads missing rows from
            # this memory at random offsets); where the kernel grants none the
            # advice changes nothing
            try:
                self._mm.madvise(mmap.MADV_HUGEPAGE)
            except OSError:
                pass
        self.array = np.frombuffer(self._mm, dtype=np.uint8)
        self.ptr = self.array.ctypes.data
        rc = torch._C._cudart.cudaHostRegister(self.ptr, self.nbytes, 3)  # portable|mapped
        if int(rc) != 0:
            raise RuntimeError(f"cudaHostRegister failed: {rc}")
        self._registered = True

    def close(self):
        if getattr(self, "_registered", False):
            import torch
            torch._C._cudart.cudaHostUnregister(self.ptr)
            self._registered = False
        self.array = None
        if getattr(self, "_mm", None) is not None:
            try:
                self._mm.close()
            except BufferError:
                pass
            self._mm = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Pool:
    """A dhs pool with its four device arenas allocated by torch."""

    def __init__(self, *, max_requests, sources, row_bytes, page_rows, tail_rows,
                 hot_rows, max_queries, max_topk, max_rows_per_request,
                 optional_pages, admission_reserve_pages=0, device=None,
                 stream=None):
        import torch
        self.device = torch.device(device or "cuda")
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.stream = stream or torch.cuda.current_stream(self.device)
        cfg = dhs_pool_config()
        cfg.max_requests, cfg.sources, cfg.row_bytes = max_requests, sources, row_bytes
        cfg.page_rows, cfg.tail_rows, cfg.hot_rows = page_rows, tail_rows, hot_rows
        cfg.max_queries, cfg.max_topk = max_queries, max_topk
        cfg.max_rows_per_request = max_rows_per_request
        cfg.optional_pages = optional_pages
        cfg.admission_reserve_pages = admission_reserve_pages
        sizes = dhs_pool_bytes(cfg)
        self.buffers = [torch.empty(max(s, 256), dtype=torch.uint8, device=self.device)
                        for s in sizes]
        cfg.hot_dev, cfg.tail_dev, cfg.opt_dev, cfg.meta_dev = [
            b.data_ptr() for b in self.buffers]
        cfg.stream = self.stream.cuda_stream
        self.cfg = cfg
        self.pages_max = -(-max_rows_per_request // page_rows)
        with torch.cuda.device(self.device):
            self.h = dhs_pool_create(cfg)

    @property
    def hot(self):
        return self.buffers[DHS_BUF_HOT]

    @property
    def tail(self):
        return self.buffers[DHS_BUF_TAIL]

    @property
    def opt(self):
        return self.buffers[DHS_BUF_OPT]

    def close(self):
        if getattr(self, "h", None):
            self.stream.synchronize()
            dhs_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def admit(self, req, src, host_ptr, n_rows, mask=None):
        return dhs_admit(self.h, req, src, host_ptr, n_rows, mask)

    def reclaim(self, order, deficit):
        return dhs_reclaim(self.h, order, deficit)

    def release(self, req):
        return dhs_release(self.h, req)

    def admit_device(self, req, src, dev_ptr, host_ptr, n_rows, mask=None):
        return dhs_admit_device(self.h, req, src, dev_ptr, host_ptr, n_rows, mask)

    def admit_window(self, req, src, dev_ptr, n_rows):
        return dhs_admit_window(self.h, req, src, dev_ptr, n_rows)

    def backup(self, max_pages):
        return dhs_backup(self.h, max_pages)

    def refill(self, max_pages):
        return dhs_refill(self.h, max_pages)

    def pending_backup(self):
        return int(lib.dhs_pending_backup(self.h))

    def used(self):
        return dhs_pool_used(self.h)

    def flush(self):
        return dhs_flush(self.h)

    def append(self, items):
        return dhs_append(self.h, items)

    def resolve(self, st):
        return dhs_resolve(self.h, st)

    def gather(self, st):
        return dhs_gather(self.h, st)

    def resolve_gather(self, st):
        return dhs_resolve_gather(self.h, st)

    def status(self):
        return dhs_status(self.h)

    def set_option(self, key, value):
        return check(dhs_set_option(self.h, key, value), "dhs_set_option")

    def get_option(self, key):
        rc, v = dhs_get_option(self.h, key)
        check(rc, "dhs_get_option")
        return v

    def read_state(self, req, src):
        return dhs_read_state(self.h, req, src, self.cfg.hot_rows, self.pages_max)

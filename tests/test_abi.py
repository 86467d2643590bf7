"""The C ABI without a GPU: libdhs.so builds for sm_103a, loads, exports every
function include/dhs.h declares, and its host-only calls (sizes, validation,
error strings) behave as documented.  No device work is issued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dhs():
    from hierarchical_sparse_kv_dhs_gb300.build import build
    build()
    from hierarchical_sparse_kv_dhs_gb300 import dhs as mod
    return mod


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dhs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dhs_[a-z_]+)\s*\(", text)) - {"dhs_pool_config"})


def test_every_declared_symbol_is_exported(dhs):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(dhs.lib, n), f"{n} declared in dhs.h but not exported"


def test_strerror(dhs):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -99):
        s = dhs.lib.dhs_strerror(code)
        assert isinstance(s, bytes) and s


def _cfg(dhs, **kw):
    c = dhs.dhs_pool_config()
    c.max_requests, c.sources, c.row_bytes, c.page_rows = 8, 4, 1152, 64
    c.tail_rows, c.hot_rows, c.max_queries, c.max_topk = 256, 4096, 1, 2048
    c.max_rows_per_request, c.optional_pages = 32832, 16384
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_pool_bytes(dhs):
    sizes = dhs.dhs_pool_bytes(_cfg(dhs))
    assert sizes[dhs.DHS_BUF_HOT] == 8 * 4 * 4096 * 1152
    assert sizes[dhs.DHS_BUF_TAIL] == 8 * 4 * 256 * 1152
    assert sizes[dhs.DHS_BUF_OPT] == 16384 * 64 * 1152
    # tags + stamps + page maps + miss lists dominate the metadata
    pairs, pmax = 32, -(-32832 // 64)
    assert sizes[dhs.DHS_BUF_META] >= pairs * (4096 * 8 + pmax * 4 + 2048 * 8)


@pytest.mark.parametrize("field,value", [
    ("row_bytes", 1000), ("page_rows", 48), ("hot_rows", 0), ("hot_rows", 20000),
    ("tail_rows", 0), ("max_requests", 0), ("admission_reserve_pages", 99999),
    ("max_rows_per_request", 0)])
def test_invalid_geometry_rejected_on_host(dhs, field, value):
    out = (ctypes.c_size_t * 4)()
    assert dhs.lib.dhs_pool_bytes(ctypes.byref(_cfg(dhs, **{field: value})), out) == dhs.DHS_EINVAL
    h = ctypes.c_void_p()
    assert dhs.lib.dhs_pool_create(ctypes.byref(_cfg(dhs, **{field: value})),
                                   ctypes.byref(h)) == dhs.DHS_EINVAL


def test_hot_cache_size_limit(dhs):
    """16384 hot slots per (request, source) is the largest B the resolve
    kernel's 16-bit slot lists take."""
    out = (ctypes.c_size_t * 4)()
    assert dhs.lib.dhs_pool_bytes(ctypes.byref(_cfg(dhs, hot_rows=16384)), out) == 0
    assert dhs.lib.dhs_pool_bytes(ctypes.byref(_cfg(dhs, hot_rows=16385)), out) == dhs.DHS_EINVAL


def test_null_arguments(dhs):
    assert dhs.lib.dhs_pool_create(None, None) == dhs.DHS_EINVAL
    h = ctypes.c_void_p()
    # valid geometry but null device buffers
    assert dhs.lib.dhs_pool_create(ctypes.byref(_cfg(dhs)), ctypes.byref(h)) == dhs.DHS_EINVAL
    assert dhs.lib.dhs_status(None, None) == dhs.DHS_EINVAL
    assert dhs.lib.dhs_flush(None) == dhs.DHS_EINVAL
    assert dhs.lib.dhs_pool_used(None) == -1
    dhs.lib.dhs_pool_destroy(None)
    # every other entry point refuses a null pool before touching a device
    n64 = ctypes.c_int64(0)
    E = dhs.DHS_EINVAL
    assert dhs.lib.dhs_admit(None, 0, 0, None, 0, None, ctypes.byref(n64)) == E
    assert dhs.lib.dhs_admit_device(None, 0, 0, None, None, 0, None, ctypes.byref(n64)) == E
    assert dhs.lib.dhs_reclaim(None, None, 0, 0, ctypes.byref(n64)) == E
    assert dhs.lib.dhs_release(None, 0) == E
    assert dhs.lib.dhs_backup(None, 1, ctypes.byref(n64)) == E
    assert dhs.lib.dhs_refill(None, 1, ctypes.byref(n64)) == E
    assert dhs.lib.dhs_pending_backup(None) == -1
    assert dhs.lib.dhs_append(None, None, 0) == E
    for fn in ("dhs_resolve", "dhs_gather", "dhs_resolve_gather", "dhs_resolve_noalloc"):
        assert getattr(dhs.lib, fn)(None, None) == E, fn
    assert dhs.lib.dhs_decode_step(None, None, 0, None) == E
    assert dhs.lib.dhs_decode_step_host(None, None, 0, None, 0, None, None, 0) == E
    assert dhs.lib.dhs_decode_step_host_async(None, None, 0, None, None, 0, None, None, 0,
                                              None) == E
    assert dhs.lib.dhs_prefetch(None, None, None) == E
    assert dhs.lib.dhs_gather_on(None, None, None) == E
    assert dhs.lib.dhs_set_option(None, dhs.DHS_OPT_EARLY, 1) == E
    assert dhs.lib.dhs_get_option(None, dhs.DHS_OPT_EARLY, ctypes.byref(n64)) == E
    assert dhs.lib.dhs_read_state(None, 0, 0, None, None, None, None) == E


def test_binding_constants_match_the_header():
    """Every integer constant include/dhs.h defines has the same value in the
    Python binding (options, item flags, error codes, status flags)."""
    import re
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    with open(os.path.join(ROOT, "include", "dhs.h")) as f:
        text = f.read()
    defs = dict(re.findall(r"^#define\s+(DHS_[A-Z0-9_]+)\s+\(?(-?(?:0x)?[0-9A-Fa-f]+)u?\)?\s*(?:/\*.*)?$",
                           text, flags=re.M))
    assert len(defs) > 20
    missing, wrong = [], []
    for name, v in defs.items():
        want = int(v, 0)
        if not hasattr(dhs, name):
            missing.append(name)
        elif getattr(dhs, name) != want:
            wrong.append((name, getattr(dhs, name), want))
    assert not wrong, wrong
    assert not missing, missing

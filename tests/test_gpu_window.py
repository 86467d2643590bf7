"""Window sources through the C ABI against the CPU oracle.

A window source ("Adaptive DHiSparse", How it works / Speculative state: a
drafter retains only the rows its window covers, stored as a ring) keeps its last
T rows, in the tail ring: no host copy, no optional pages, no hot cache.
Pools here mix window sources with ordinary ones, and every decode step
appends rows to both and resolves + gathers verify blocks of two queries
(k = 24, not a multiple of a gather tile).  Window selections stay inside
the window except on some steps, which must fail with ERANGE while their
in-window entries keep their locations.  Locations, counters, status flags,
hot-cache state and every staged byte must match the oracle exactly, fused
and split, with either gather, early copies on and off.
"""
import ctypes

import numpy as np
import pytest
import torch

import dhs_workload

pytestmark = pytest.mark.gpu

TAG = 95
E = 576
R, S, Q, K = 2, 2, 2, 24
N_ORD = 700  # ordinary sources' imported rows (10 complete pages of 64, one partial)
MAX_ROWS = 1200


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hierarchical_sparse_kv_dhs_gb300.build import build
    import oracle
    build()
    oracle.build()
    dhs_workload.build()


def payload(r, s, row0, n):
    return dhs_workload.payload_rows(TAG, s, r, row0, n, E)


def run_window_pool(T, mode, steps=12, seed=0, union=False, how="plain"):
    """how: "plain" (dhs_decode_step when fused, else append + resolve +
    gather), "prefetch" (resolves by dhs_prefetch on a side stream, then the
    gather) or "noalloc" (resolves by dhs_resolve_noalloc)."""
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    from oracle import OraclePool
    rng = np.random.default_rng(seed)
    B = 64
    pool = dhs.Pool(max_requests=R, sources=S, row_bytes=E * 2, page_rows=64, tail_rows=T,
                    hot_rows=B, max_queries=Q, max_topk=K, max_rows_per_request=MAX_ROWS,
                    optional_pages=16)
    host = dhs.HostRows(R * S * MAX_ROWS * E * 2)
    orc = OraclePool(R, S, T, B, E, 64, MAX_ROWS, 16)
    fused, impl, early = mode
    pool.set_option(dhs.DHS_OPT_GATHER_IMPL, impl)
    pool.set_option(dhs.DHS_OPT_EARLY, early)
    # source 0 of each request ordinary (half its pages resident), source 1 a window
    L = {}
    keep = []
    for r in range(R):
        off = (r * S) * MAX_ROWS * E * 2
        rows = payload(r, 0, 0, N_ORD)
        host.array[off: off + rows.nbytes] = rows.view(np.uint8).ravel()
        mask = (np.arange(N_ORD // 64) % 2 == 0).astype(np.uint8)
        assert pool.admit(r, 0, host.ptr + off, N_ORD, mask)[0] == 0
        assert orc.admit(r, 0, N_ORD, mask, rows) == (0, 0)
        L[(r, 0)] = N_ORD
        n = int(rng.integers(0, 3 * T))
        m = min(n, T)
        win = payload(r, 1, n - m, m)
        dev = torch.from_numpy(win.view(np.int16).copy()).cuda()
        keep.append(dev)
        assert pool.admit_window(r, 1, dev.data_ptr() if m else None, n) == 0
        assert orc.admit_window(r, 1, n, win) == 0
        L[(r, 1)] = n
    assert pool.used() == orc.used()
    sel_d = torch.zeros((R, S, Q, K), dtype=torch.int32, device="cuda")
    loc_d = torch.zeros((R, S, Q, K), dtype=torch.int32, device="cuda")
    cnt_d = torch.zeros((R, S, 8), dtype=torch.int32, device="cuda")
    idx_d = torch.zeros((R, S, Q, K), dtype=torch.int32, device="cuda")
    stg_d = torch.zeros((R, S, Q, K, E), dtype=torch.int16, device="cuda")
    items = []
    for r in range(R):
        for s in range(S):
            it = dhs.dhs_item()
            it.req, it.src, it.queries, it.topk = r, s, Q, K
            it.sel_dev = sel_d[r, s].data_ptr()
            it.loc_dev = loc_d[r, s].data_ptr()
            it.counters_dev = cnt_d[r, s].data_ptr()
            it.staging_dev = stg_d[r, s].data_ptr()
            if union:
                it.flags = dhs.DHS_ITEM_UNION
                it.index_dev = idx_d[r, s].data_ptr()
            items.append(it)
    erange_steps = 0
    try:
        for step in range(1, steps + 1):
            # appends: 0 .. T rows per source
            apps, app_keep = [], []
            for r in range(R):
                for s in range(S):
                    a = int(rng.integers(0, min(T, 3) + 1))
                    if L[(r, s)] + a > MAX_ROWS - 1:
                        a = 0
                    rows = payload(r, s, L[(r, s)], a)
                    if a:
                        dev = torch.from_numpy(rows.view(np.int16).copy()).cuda()
                        app_keep.append(dev)
                        it = dhs.dhs_append_item()
                        it.req, it.src, it.count, it.rows_dev = r, s, a, dev.data_ptr()
                        apps.append(it)
                        assert orc.append(r, s, a, rows) == 0
                    L[(r, s)] += a
            # selections
            sel = np.zeros((R, S, Q, K), np.int32)
            bad = step % 4 == 3
            for r in range(R):
                sel[r, 0] = rng.integers(0, L[(r, 0)], size=(Q, K))
                lo, hi = max(0, L[(r, 1)] - T), L[(r, 1)]
                if hi == 0:
                    sel[r, 1] = 0  # empty window: every row is out of range
                else:
                    sel[r, 1] = rng.integers(lo, hi, size=(Q, K))
                if bad and r == 1:  # one row just below the window (or beyond L)
                    sel[r, 1, 1, 5] = lo - 1 if lo > 0 else hi
            sel_d.copy_(torch.from_numpy(sel))
            st, arr = dhs.make_step(step, items)
            if how == "prefetch":
                if apps:
                    assert dhs.dhs_append(pool.h, apps) == 0
                side = torch.cuda.Stream()
                assert dhs.lib.dhs_prefetch(pool.h, ctypes.byref(st),
                                            ctypes.c_void_p(side.cuda_stream)) == 0
                assert dhs.dhs_gather(pool.h, st) == 0
            elif how == "noalloc":
                if apps:
                    assert dhs.dhs_append(pool.h, apps) == 0
                assert dhs.lib.dhs_resolve_noalloc(pool.h, ctypes.byref(st)) == 0
                assert dhs.dhs_gather(pool.h, st) == 0
            elif fused:
                assert dhs.dhs_decode_step(pool.h, apps, st) == 0
            else:
                if apps:
                    assert dhs.dhs_append(pool.h, apps) == 0
                assert dhs.dhs_resolve(pool.h, st) == 0
                assert dhs.dhs_gather(pool.h, st) == 0
            torch.cuda.synchronize()
            rc, flags = pool.status()
            want_flags = 0
            loc = loc_d.cpu().numpy().view(np.uint32)
            cnt = cnt_d.cpu().numpy().view(np.uint32)
            idx = idx_d.cpu().numpy()
            stg = stg_d.cpu().numpy().view(np.uint16)
            for r in range(R):
                for s in range(S):
                    if union:
                        orc_rc, oloc, oidx, ocnt = orc.resolve_union(step, r, s, sel[r, s])
                        assert np.array_equal(idx[r, s], oidx), (mode, step, r, s)
                        oloc = oloc.reshape(Q, K)
                    else:
                        orc_rc, oloc, ocnt = orc.resolve(step, r, s, sel[r, s])
                    if orc_rc == "erange":
                        want_flags |= 1
                        erange_steps += s == 1
                    assert np.array_equal(loc[r, s], oloc), (mode, step, r, s)
                    assert np.array_equal(cnt[r, s], ocnt), (mode, step, r, s, cnt[r, s], ocnt)
                    if union:  # the distinct rows staged once, in row order
                        u = int(ocnt[1])
                        grc, ostg = orc.gather(oloc.ravel()[:u])
                        assert grc == 0
                        got = stg[r, s].reshape(Q * K, E)[:u]
                        assert np.array_equal(got, ostg), (mode, step, r, s)
                    else:
                        grc, ostg = orc.gather(oloc)
                        assert grc == 0
                        assert np.array_equal(stg[r, s], ostg), (mode, step, r, s)
                    tags, stamps, pages, info = pool.read_state(r, s)
                    ot, os_, op, ln = orc.state(r, s)
                    assert np.array_equal(tags, ot) and np.array_equal(stamps, os_)
                    assert np.array_equal(pages, op) and int(info[1]) == ln[1]
                    if s == 1:
                        assert (tags == -1).all() and (pages == -1).all() and int(info[0]) == 0
            assert flags == want_flags, (mode, step, flags, want_flags)
        assert erange_steps >= 2
        # the window sources' payload bytes never reached host memory
        for r in range(R):
            off = (r * S + 1) * MAX_ROWS * E * 2
            assert not host.array[off: off + MAX_ROWS * E * 2].any()
    finally:
        pool.close()
        host.close()
        orc.close()


MODES = {"fused-tma": (True, 1, 1), "fused-vec": (True, 0, 1), "fused-tma-late": (True, 1, 0),
         "split-tma": (False, 1, 1), "split-vec": (False, 0, 1)}


@pytest.mark.parametrize("T", [1, 16, 64])
@pytest.mark.parametrize("mode", list(MODES))
def test_window_sources_match_oracle(T, mode):
    run_window_pool(T, MODES[mode], seed=T)


@pytest.mark.parametrize("how", ["union-fused", "union-split", "prefetch", "noalloc"])
def test_window_sources_other_entry_points(how):
    """Window sources under union staging (fused and split), resolved by
    dhs_prefetch on a side stream, and by dhs_resolve_noalloc."""
    if how.startswith("union"):
        run_window_pool(16, (how == "union-fused", 1, 1), seed=7, union=True)
    else:
        run_window_pool(16, (False, 1, 1), seed=8, how=how)


def test_window_golden_trace_gpu():
    from fixture_runner import run_trace
    from gpu_adapter import GpuAdapter
    run_trace("window_micro.txt", GpuAdapter(), elems=8)


def test_admit_window_rejects_bad_arguments():
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    pool = dhs.Pool(max_requests=1, sources=1, row_bytes=64, page_rows=4, tail_rows=4,
                    hot_rows=4, max_queries=1, max_topk=4, max_rows_per_request=16,
                    optional_pages=0)
    rows = torch.zeros(64, dtype=torch.uint8, device="cuda")
    try:
        assert pool.admit_window(0, 0, None, 3) == dhs.DHS_EINVAL       # rows missing
        assert pool.admit_window(0, 0, rows.data_ptr() + 8, 1) == dhs.DHS_EINVAL  # misaligned
        assert pool.admit_window(0, 0, rows.data_ptr(), 17) == dhs.DHS_EINVAL     # too long
        assert pool.admit_window(0, 1, rows.data_ptr(), 1) == dhs.DHS_EINVAL      # no source 1
        assert pool.admit_window(0, 0, rows.data_ptr(), 1) == dhs.DHS_OK
        assert pool.admit_window(0, 0, rows.data_ptr(), 1) == dhs.DHS_ESTATE
        torch.cuda.synchronize()
    finally:
        pool.close()

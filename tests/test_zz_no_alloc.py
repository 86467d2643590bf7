"""dhs_resolve_noalloc against dhs_resolve, through the C ABI.

dhs_resolve_noalloc serves callers that cannot allocate device memory where
they resolve (an embedding runtime that hands the library only its own
buffers, or code running where allocation calls are not permitted): it keeps
the per-item miss lists in a fixed device array inside libdhs.so instead of
the pool's metadata buffer.  Two identical pools run the same two decode
steps, one through each entry point; locations, counters, hot-cache state and
gathered bytes must be identical (the path is integer and byte work:
bit-exact), on both calls in a row.  The workload keeps the hot cache busy
(low residency, small B) so the miss lists and the host copy are exercised.

Kept in its own file, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hierarchical_sparse_kv_dhs_gb300.build import build
    import dhs_workload
    build()
    dhs_workload.build()
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    f = dhs.lib.dhs_resolve_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.POINTER(dhs.dhs_step)]
    return dhs


def _same_results(cfg, ref, new):
    torch.cuda.synchronize()
    assert ref.status() == (0, 0) and new.status() == (0, 0)
    assert torch.equal(ref.loc, new.loc)
    assert torch.equal(ref.counters, new.counters)
    assert torch.equal(ref.staging.view(torch.int16), new.staging.view(torch.int16))
    for r in range(cfg.requests):
        for s in range(cfg.sources):
            a, b = ref.pool.read_state(r, s), new.pool.read_state(r, s)
            assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert ref.counters[..., 5].sum().item() > 0, "the workload must fetch rows from host"


def _resolve_noalloc(dhs, run, step):
    st, _ = run._steps[step - 1]
    assert dhs.lib.dhs_resolve_noalloc(run.pool.h, ctypes.byref(st)) == dhs.DHS_OK


def test_noalloc_resolve_matches_resolve_two_calls(lib):
    """Two identical pools, two decode steps, one pool resolved through each
    entry point.  Between the two steps another pool, with more (request,
    source) pairs and longer miss lists (so the fixed array is laid out
    differently), resolves through the no-allocation entry point on the same
    stream: it overwrites the shared array, and the first pool's second step
    must still match, since every entry a call reads it wrote itself."""
    dhs = lib
    from dhs_workload.configs import TINY, Workload
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun

    cfg = TINY.scaled(name="noalloc", tag=71, requests=3, sources=2, residency=0.1,
                      hot=300, steps=2)
    other_cfg = TINY.scaled(name="noalloc_other", tag=72, requests=5, sources=2,
                            residency=0.0, hot=500, topk=400, steps=1)
    wl, other_wl = Workload(cfg), Workload(other_cfg)
    ref, new = GpuRun(cfg, wl), GpuRun(cfg, wl)
    other_ref, other = GpuRun(other_cfg, other_wl), GpuRun(other_cfg, other_wl)
    assert new.pool.stream.cuda_stream == other.pool.stream.cuda_stream
    try:
        for step in (1, 2):
            ref.append(step)
            new.append(step)
            ref.resolve(step)
            _resolve_noalloc(dhs, new, step)
            ref.gather(step)
            new.gather(step)
            _same_results(cfg, ref, new)
            if step == 1:
                other_ref.append(1)
                other.append(1)
                other_ref.resolve(1)
                _resolve_noalloc(dhs, other, 1)
                other_ref.gather(1)
                other.gather(1)
                _same_results(other_cfg, other_ref, other)
    finally:
        for run in (ref, new, other_ref, other):
            run.close()


def test_noalloc_rejects_pools_beyond_the_limit(lib):
    dhs = lib
    # 64 x 4 pairs x min(4096, 2048) = 524288 miss entries > 65536
    pool = dhs.Pool(max_requests=64, sources=4, row_bytes=1152, page_rows=64,
                    tail_rows=16, hot_rows=4096, max_queries=1, max_topk=2048,
                    max_rows_per_request=4096, optional_pages=0)
    st, keep = dhs.make_step(1, [])
    try:
        assert dhs.lib.dhs_resolve_noalloc(pool.h, ctypes.byref(st)) == dhs.DHS_EINVAL
    finally:
        pool.close()

"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Small configurations (every request, every step, every output): locations,
counters, hot-cache tags and stamps, page maps, gathered bytes, and the
written-through host rows must be identical -- the path is integer and byte
work, so the bar is bit-exact.  The hand-worked golden traces run through
the library too.  Full-size workloads run every request on the GPU in the
launch configuration the benchmark times, and compare a sample of requests
against the oracle (requests are independent once admitted, so the sampled
ones are exact), plus properties of every request.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from dhs_workload.configs import C8, C64, C128, LONG, TINY, Config, Workload  # noqa: E402
from fixture_runner import run_trace  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hierarchical_sparse_kv_dhs_gb300.build import build
    import oracle
    import dhs_workload
    build()
    oracle.build()
    dhs_workload.build()


def _as_u32(t):
    return t.cpu().numpy().view(np.uint32)


def compare_run(cfg: Config, sampled=None, check_all_bytes=True, fused=True,
                gather_impl=0, patch=None, early=1, union=False, fresh=None, tpc=None,
                stage=None, polls=None, copy_pdl=None, copy_ctas=None, resolve_paired=None,
                steal=None, resolve_ctas=None):
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    from oracle.run import OracleRun
    wl = Workload(cfg)
    if patch:
        patch(wl)
    big = cfg.pairs * cfg.max_rows * cfg.row_bytes > (8 << 30)
    gpu = GpuRun(cfg, wl, gather_impl=gather_impl,
                 payload_requests=sampled if (big and sampled is not None) else None,
                 union=union)
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    if early != 1:
        gpu.pool.set_option(dhs.DHS_OPT_EARLY, early)
    if fresh is not None:
        gpu.pool.set_option(dhs.DHS_OPT_FRESH_LIST, fresh)
    if tpc is not None:
        gpu.pool.set_option(dhs.DHS_OPT_GATHER_TPC, tpc)
    if stage is not None:
        gpu.pool.set_option(dhs.DHS_OPT_STAGE_MISSES, stage)
    if polls is not None:
        gpu.pool.set_option(dhs.DHS_OPT_MARK_POLLS, polls)
    if copy_pdl is not None:
        gpu.pool.set_option(dhs.DHS_OPT_COPY_PDL, copy_pdl)
    if copy_ctas is not None:
        gpu.pool.set_option(dhs.DHS_OPT_COPY_CTAS, copy_ctas)
    if resolve_paired is not None:
        gpu.pool.set_option(dhs.DHS_OPT_RESOLVE_PAIRED, resolve_paired)
    if steal is not None:
        gpu.pool.set_option(dhs.DHS_OPT_COPY_STEAL, steal)
    if resolve_ctas is not None:
        gpu.pool.set_option(dhs.DHS_OPT_RESOLVE_CTAS, resolve_ctas)
    sampled = list(range(cfg.requests)) if sampled is None else sampled
    orc = OracleRun(cfg, wl, requests=sampled, union=union)
    try:
        for r in sampled:
            for s in range(cfg.sources):
                g_pages = gpu.pool.read_state(r, s)[2]
                o_pages = orc.pool.state(r, s)[2]
                assert np.array_equal(g_pages, o_pages), (r, s)
        assert gpu.pool.used() == orc.pool.used()
        for step in range(1, cfg.total_steps + 1):
            gpu.step(step, fused=fused)
            res = orc.step(step)
            rc, flags = gpu.status()
            want_flags = 0
            for r in sampled:
                for s in range(cfg.sources):
                    want_flags |= {0: 0, "erange": 1, "ebudget": 2}[res[r]["rc"][s]]
            if len(sampled) == cfg.requests:
                assert flags == want_flags, (step, rc, flags, want_flags)
            else:
                assert (flags & ~3) == 0 and (flags & want_flags) == want_flags
            loc_all = _as_u32(gpu.loc)
            cnt_all = _as_u32(gpu.counters)
            idx_all = gpu.index.cpu().numpy() if union else None
            for r in sampled:
                o = res[r]
                assert np.array_equal(loc_all[r].reshape(cfg.sources, -1),
                                      o["loc"].reshape(cfg.sources, -1)), (cfg.name, step, r)
                assert np.array_equal(cnt_all[r], o["counters"]), \
                    (cfg.name, step, r, cnt_all[r], o["counters"])
                stg = gpu.staging[r].cpu().view(torch.int16).numpy().view(np.uint16)
                if union:
                    assert np.array_equal(idx_all[r], o["index"]), (cfg.name, step, r)
                    for layer, want in enumerate(o["staging"]):
                        got = stg[layer].reshape(-1, cfg.row_elems)[: len(want)]
                        if not check_all_bytes and len(want):
                            pick = np.linspace(0, len(want) - 1, 67).astype(int)
                            got, want = got[pick], want[pick]
                        assert np.array_equal(got, want), (cfg.name, step, r, layer)
                elif check_all_bytes:
                    assert np.array_equal(stg, o["staging"]), (cfg.name, step, r)
                else:
                    idx = np.linspace(0, cfg.topk - 1, 67).astype(int)
                    assert np.array_equal(stg[:, :, idx], o["staging"][:, :, idx])
                for s in range(cfg.sources):
                    gt, gs, _, info = gpu.pool.read_state(r, s)
                    ot, os_, _, ln = orc.pool.state(r, s)
                    assert np.array_equal(gt, ot) and np.array_equal(gs, os_), (step, r, s)
                    assert int(info[1]) == ln[1]
            # every request: counters add up, scan bounded by B
            c = cnt_all.reshape(-1, 8)
            assert (c[:, 2] + c[:, 3] + c[:, 4] + c[:, 5] == c[:, 1]).all()
            assert (c[:, 6] <= cfg.hot).all()
        # written-through host rows of the sampled pairs
        for r in sampled:
            for s in range(cfg.sources):
                L = wl.length(r, cfg.total_steps)
                got = gpu.host_rows(r, s, 0, L)
                want = orc.pool.rows(r, s, 0, 0, L)
                assert np.array_equal(got, want), (r, s)
    finally:
        gpu.close()
        orc.pool.close()


# ------------------------------------------------------------ golden traces

@pytest.mark.parametrize("trace", ["resolve_micro_b2.txt", "resolve_micro_b3_pairs.txt",
                                   "admission_micro.txt", "backup_refill_micro.txt",
                                   "resolve_micro_same_step.txt"])
def test_golden_trace_gpu(trace):
    from gpu_adapter import GpuAdapter
    run_trace(trace, GpuAdapter(), elems=8)  # 16-byte rows


@pytest.mark.parametrize("seed", range(12))
def test_admission_sequences_match_oracle(seed):
    """Device admission, deferred backup, reclaim, release, refill, appends
    and resolves in random order: the library and the oracle agree on every
    result, page map and host row, and every gathered row is its payload."""
    from admission_seq import run_sequence
    from fixture_runner import OracleAdapter
    from gpu_adapter import GpuAdapter
    run_sequence([OracleAdapter(), GpuAdapter()], seed, reserve=seed % 3)


@pytest.mark.parametrize("residency", [True, False])
def test_loadstep_matches_oracle(residency):
    """The load-step schedule (admission pressure rising and draining, with
    reclaim, deferred backup and refill) through the library and the
    oracle: every step's results, locations and counters agree, and every
    gathered row on the GPU is its payload."""
    from dhs_workload.loadstep import LOADSTEP_SMALL, LoadStepInputs, run
    from fixture_runner import OracleAdapter
    from gpu_adapter import GpuAdapter
    cfg = LOADSTEP_SMALL
    got, want = {}, {}

    def keep(into):
        return lambda step, res: into.__setitem__(step, res)

    gpu = GpuAdapter(max_queries=1, max_topk=cfg.topk)
    rec_g = run(gpu, cfg, residency, LoadStepInputs(cfg), keep(got))
    rec_o = run(OracleAdapter(), cfg, residency, LoadStepInputs(cfg), keep(want))
    assert rec_g == rec_o
    inputs = LoadStepInputs(cfg)
    for step in want:
        for (r, s, rc, loc, cnt, sel), (r2, s2, rc2, loc2, cnt2, _) in zip(want[step], got[step]):
            assert (r, s, rc) == (r2, s2, rc2)
            assert np.array_equal(np.asarray(loc).ravel(), np.asarray(loc2).ravel()), (step, r, s)
            assert np.array_equal(np.asarray(cnt), np.asarray(cnt2)), (step, r, s)
    # byte truth of the last step's gathers on the GPU
    step = max(got)
    for r, s, rc, loc, cnt, sel in got[step]:
        st = gpu.gather(np.asarray(loc).ravel())
        for e in range(0, len(sel), 7):
            assert np.array_equal(st[e], inputs.rows(r, s, int(sel[e]), 1)[0]), (r, s, e)


# ------------------------------------------------------------ small, every output

SMALL = [
    TINY,
    # verify block of 3 queries, speculative appends, ragged k (not a tile multiple)
    TINY.scaled(name="v3", tag=41, queries=3, topk=77, verify_core=50, hot=300,
                steps=10, append_lo=1, append_hi=4, requests=3, sources=2),
    # Reuse layers with a shared selection over 3 sources, low residency
    TINY.scaled(name="reuse", tag=42, requests=3, sources=3, reuse_layers=3,
                shared_selection=True, residency=0.2, steps=8, hot=700),
    # admission-driven residency under capacity pressure, temporal locality
    TINY.scaled(name="pressure", tag=43, requests=6, sources=2, residency=None,
                capacity_frac=0.3, rho=0.9, steps=12, warmup_steps=4, hot=256),
    # tiny hot cache: heavy eviction every step
    TINY.scaled(name="evict", tag=44, requests=2, sources=1, hot=200, topk=150,
                residency=0.0, steps=12),
    # non-1152-byte rows (generic gather/copy paths), short tail, 2 sources
    TINY.scaled(name="rows", tag=45, row_elems=200, tail=5, requests=2, sources=2,
                steps=6, topk=100),
]


IMPLS = {"vec": 0, "tma": 1}


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
@pytest.mark.parametrize("mode", ["fused-vec", "fused-tma", "split-vec", "split-tma",
                                  "fused-tma-late", "fused-vec-late", "prefetch-tma"])
def test_small_configs_bit_exact(cfg, mode):
    fused = "prefetch" if mode.startswith("prefetch") else mode.startswith("fused")
    compare_run(cfg, fused=fused, gather_impl=IMPLS[mode.split("-")[1]],
                early=0 if mode.endswith("late") else 1)


UNION = [SMALL[1], SMALL[2], SMALL[4],
         TINY.scaled(name="v8", tag=49, queries=8, verify_core=40, topk=64, hot=400,
                     steps=8, append_lo=1, append_hi=8, requests=2, sources=2,
                     residency=0.3)]


@pytest.mark.parametrize("cfg", UNION, ids=[c.name for c in UNION])
@pytest.mark.parametrize("mode", ["fused-tma", "fused-vec", "split-tma"])
def test_union_staging_bit_exact(cfg, mode):
    compare_run(cfg, fused=mode.startswith("fused"), gather_impl=IMPLS[mode.split("-")[1]],
                union=True)


# five Reuse layers on one location vector: the host copy writes the fetched
# rows of three of them, the other two take the fresh-row list
REUSE5 = TINY.scaled(name="reuse5", tag=54, requests=2, sources=2, reuse_layers=5,
                     shared_selection=True, residency=0.2, steps=6, hot=700)


@pytest.mark.parametrize("cfg", [SMALL[1], SMALL[2], SMALL[4], UNION[3], REUSE5],
                         ids=["v3", "reuse", "evict", "v8", "reuse5"])
def test_misses_staged_by_the_host_copy_or_not(cfg):
    """Fused steps: the host copy writes the rows it fetches into the
    resolved items' staging and that of up to three Reuse items sharing
    their locations (default), or leaves them to the gather."""
    for stage in (1, 0):
        compare_run(cfg, gather_impl=1, stage=stage)
        compare_run(cfg, gather_impl=1, stage=stage, union=True)
        compare_run(cfg, gather_impl=1, stage=stage, fresh=0)


# fully resident: every resolved item's rows resolve in step 1, so an item
# publishes its location mark only because Reuse items read its vector
RESIDENT_REUSE = TINY.scaled(name="resident_reuse", tag=55, requests=2, sources=2,
                             reuse_layers=3, shared_selection=True, residency=1.0, steps=6)


def test_location_mark_of_step1_only_items_read_by_reuse_items():
    """An item whose rows all resolve in step 1 leaves its location mark out
    unless a gather-only item of the launch reads its vector.  Here Reuse
    items read such vectors: the results are bit-exact, and no step waits
    for a gather tile's bounded poll to run out (about a second) before it
    falls back to waiting for the grids."""
    import time
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    cfg = RESIDENT_REUSE
    compare_run(cfg, gather_impl=1)
    run = GpuRun(cfg, Workload(cfg), gather_impl=1)
    try:
        worst = 0.0
        for step in range(1, cfg.total_steps + 1):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            run.step(step)
            torch.cuda.synchronize()
            if step > 1:
                worst = max(worst, time.perf_counter() - t0)
            # no hot-cache hits or misses: every row resolved in step 1
            assert int(run.counters[..., 4:6].sum()) == 0, step
        assert worst < 0.1, worst
    finally:
        run.close()


@pytest.mark.parametrize("cfg", SMALL + [UNION[3], REUSE5, RESIDENT_REUSE],
                         ids=[c.name for c in SMALL] + ["v8", "reuse5", "resident_reuse"])
def test_mark_poll_fallbacks(cfg):
    """Poll limit 0: no gather tile reads an item's published locations and
    no host-copy block reads an item's published miss list; every one of
    them takes the fallback of waiting for the whole resolve (and host-copy)
    grids.  The results stay bit-exact, per query and union layout, with the
    fresh-row list on and off."""
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    compare_run(cfg, gather_impl=1, polls=0)
    compare_run(cfg, gather_impl=1, polls=0, fresh=0)
    compare_run(cfg, gather_impl=1, polls=0, union=True)
    # a poll or two: marks that come late send single tiles, blocks or warps
    # (a copy warp waiting for an item's staging entries) down the fallback
    # while the others use the marks
    compare_run(cfg, gather_impl=1, polls=1)
    compare_run(cfg, gather_impl=0, polls=2, fused=False)
    # the option's range and its value in effect
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    run = GpuRun(TINY, Workload(TINY))
    try:
        h, key = run.pool.h, dhs.DHS_OPT_MARK_POLLS
        assert run.pool.get_option(key) == 1 << 20
        assert dhs.dhs_set_option(h, key, 0) == dhs.DHS_OK
        assert run.pool.get_option(key) == 0
        assert dhs.dhs_set_option(h, key, (1 << 20) + 1) == dhs.DHS_EINVAL
        assert dhs.dhs_set_option(h, key, -2) == dhs.DHS_EINVAL
        assert dhs.dhs_set_option(h, key, -1) == dhs.DHS_OK
        assert run.pool.get_option(key) == 1 << 20
    finally:
        run.close()


@pytest.mark.parametrize("cfg", SMALL + [UNION[3], REUSE5],
                         ids=[c.name for c in SMALL] + ["v8", "reuse5"])
def test_host_copy_launched_after_the_resolve_grid(cfg):
    """The host copy launched after the resolve grid instead of overlapping it
    (DHS_OPT_COPY_PDL 0, what pools with large pinned regions do), with one
    block per item and with more blocks than items: bit-exact, fused and
    split, both staging layouts."""
    items = cfg.requests * cfg.sources
    for ctas in (0, max(1, items), 3 * items + 5):
        compare_run(cfg, gather_impl=1, copy_pdl=0, copy_ctas=ctas or None)
    compare_run(cfg, gather_impl=1, copy_pdl=0, fused=False)
    compare_run(cfg, gather_impl=1, copy_pdl=0, union=True)
    compare_run(cfg, gather_impl=0, copy_pdl=0)


@pytest.mark.parametrize("cfg", SMALL + [UNION[3], REUSE5],
                         ids=[c.name for c in SMALL] + ["v8", "reuse5"])
def test_host_copy_block_sharing(cfg):
    """The host copy's blocks each copying only their own items' rows
    (DHS_OPT_COPY_STEAL 0, what launches past the translation reach do), and
    claiming rows through the per-item cursors with blocks done with their
    own items taking the others' rows (1; also with more blocks than items,
    and with the copy after the resolve grid): bit-exact, fused, split and
    side-stream prefetch, both staging layouts, both gathers."""
    items = cfg.requests * cfg.sources
    compare_run(cfg, gather_impl=1, steal=0)
    compare_run(cfg, gather_impl=1, steal=0, copy_pdl=0, union=True)
    compare_run(cfg, gather_impl=0, steal=0, fused=False)
    compare_run(cfg, gather_impl=1, steal=1, copy_ctas=3 * items + 5)
    compare_run(cfg, gather_impl=1, steal=1, copy_pdl=0, fused=False)
    compare_run(cfg, gather_impl=0, steal=1, union=True)
    compare_run(cfg, gather_impl=1, steal=1, polls=0)
    compare_run(cfg, fused="prefetch", gather_impl=1, steal=1)
    compare_run(cfg, fused="prefetch", gather_impl=1, steal=0)


@pytest.mark.parametrize("cfg", SMALL + [UNION[3], REUSE5],
                         ids=[c.name for c in SMALL] + ["v8", "reuse5"])
def test_resolve_ctas_several_items_each(cfg):
    """Fewer resolve CTAs than items (DHS_OPT_RESOLVE_CTAS): CTA b resolves
    items b, b + n, ... one after the other, publishing each item's marks as
    it goes, while the host copy and the gather run beside it.  Bit-exact,
    fused, split and side-stream prefetch, both staging layouts, both copy
    modes."""
    for ctas in (1, 3):
        compare_run(cfg, gather_impl=1, resolve_ctas=ctas)
    compare_run(cfg, gather_impl=1, resolve_ctas=2, union=True)
    compare_run(cfg, gather_impl=0, resolve_ctas=2, fused=False)
    compare_run(cfg, gather_impl=1, resolve_ctas=2, copy_pdl=0, steal=0)
    compare_run(cfg, gather_impl=1, resolve_ctas=2, resolve_paired=1, polls=0)
    compare_run(cfg, fused="prefetch", gather_impl=1, resolve_ctas=2)


def test_resolve_ctas_with_failed_items():
    """A CTA whose item fails (ERANGE, EBUDGET) goes on to its next item."""
    cfg = TINY.scaled(name="range", tag=46, requests=2, sources=2, steps=4, residency=0.6)
    compare_run(cfg, gather_impl=1, patch=_bad_row, resolve_ctas=1)
    compare_run(cfg, gather_impl=1, patch=_bad_row, resolve_ctas=3, union=True)
    cfg = TINY.scaled(name="budget", tag=47, requests=2, sources=1, hot=16, topk=64,
                      residency=0.4, steps=4)
    compare_run(cfg, gather_impl=1, resolve_ctas=1)
    cfg = TINY.scaled(name="ubudget", tag=50, requests=2, sources=1, hot=16, topk=64,
                      queries=2, verify_core=32, residency=0.0, steps=4)
    compare_run(cfg, union=True, gather_impl=1, resolve_ctas=1)


def test_resolve_ctas_option_bounds():
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    cfg = SMALL[0]
    run = GpuRun(cfg, Workload(cfg))
    try:
        h, key = run.pool.h, dhs.DHS_OPT_RESOLVE_CTAS
        assert run.pool.get_option(key) == 0
        assert dhs.dhs_set_option(h, key, 5) == dhs.DHS_OK
        assert run.pool.get_option(key) == 5
        assert dhs.dhs_set_option(h, key, -1) == dhs.DHS_EINVAL
        assert dhs.dhs_set_option(h, key, 0) == dhs.DHS_OK
    finally:
        run.close()


def test_copy_steal_option_bounds():
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    cfg = SMALL[0]
    run = GpuRun(cfg, Workload(cfg))
    try:
        h, key = run.pool.h, dhs.DHS_OPT_COPY_STEAL
        assert run.pool.get_option(key) == -1
        for v in (0, 1, -1):
            assert dhs.dhs_set_option(h, key, v) == dhs.DHS_OK
            assert run.pool.get_option(key) == v
        assert dhs.dhs_set_option(h, key, 2) == dhs.DHS_EINVAL
        assert dhs.dhs_set_option(h, key, -2) == dhs.DHS_EINVAL
    finally:
        run.close()


@pytest.mark.parametrize("tpc", [2, 5])
@pytest.mark.parametrize("cfg", [SMALL[1], SMALL[2], SMALL[4]], ids=["v3", "reuse", "evict"])
def test_gather_tiles_per_cta(cfg, tpc):
    """Several consecutive tiles per TMA gather CTA (tiles of different items
    in one CTA, a ragged last CTA): same results, fused and split, both
    staging layouts."""
    compare_run(cfg, gather_impl=1, tpc=tpc)
    compare_run(cfg, gather_impl=1, tpc=tpc, fused=False)
    compare_run(cfg, gather_impl=1, tpc=tpc, union=True)


@pytest.mark.parametrize("fresh", [0, 1])
@pytest.mark.parametrize("cfg", [SMALL[1], SMALL[2], SMALL[4]], ids=["v3", "reuse", "evict"])
def test_fresh_row_list_on_and_off(cfg, fresh):
    """Rows in hot slots the step's host copy fills either wait in their gather
    tile (0) or go to the list copied after the copy (1; the Reuse workload
    overflows the list on its first step, so tiles also take the fallback)."""
    compare_run(cfg, gather_impl=1, fresh=fresh)
    compare_run(cfg, gather_impl=1, fresh=fresh, union=True)


def test_prefetch_per_layer_pipeline_matches_oracle():
    """Every layer resolved on a side stream at step start (dhs_prefetch),
    then each layer gathered on its own just before it is needed, with other
    work on the pool's stream in between: the same results as the oracle."""
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    from oracle.run import OracleRun
    cfg = SMALL[2]  # three sources sharing a selection, three Reuse layers
    wl = Workload(cfg)
    gpu = GpuRun(cfg, wl)
    orc = OracleRun(cfg, wl)
    filler = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    try:
        for step in range(1, cfg.total_steps + 1):
            gpu.append(step)
            # layer 0 on the pool's stream, the other resolving layers on the
            # side stream; layer 0's gather runs alongside their resolve
            gpu.resolve_layer(step, 0)
            gpu.prefetch_layers(step, list(range(1, cfg.sources)))
            for layer in range(len(gpu.layers)):
                filler.add_(1)  # the caller's work between layers
                gpu.gather_layer(step, layer)
            res = orc.step(step)
            assert gpu.status() == (0, 0)
            loc = _as_u32(gpu.loc)
            for r in range(cfg.requests):
                assert np.array_equal(loc[r], res[r]["loc"]), (step, r)
                stg = gpu.staging[r].cpu().view(torch.int16).numpy().view(np.uint16)
                assert np.array_equal(stg, res[r]["staging"]), (step, r)
    finally:
        gpu.close()
        orc.pool.close()


def test_gathers_on_a_second_stream_match_oracle():
    """The pipelined schedule: layer 0 resolved on the pool's stream, the
    other resolving layers prefetched on a side stream, every layer gathered
    on a second stream (dhs_gather_on) while the caller's work for the
    previous layer runs on the pool's stream; then the next step's appends
    and resolves on the pool's stream (which must wait for those gathers)."""
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    from oracle.run import OracleRun
    cfg = SMALL[2]
    wl = Workload(cfg)
    gpu = GpuRun(cfg, wl)
    orc = OracleRun(cfg, wl)
    g = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    filler = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    try:
        for step in range(1, cfg.total_steps + 1):
            gpu.append(step)
            gpu.resolve_layer(step, 0)
            gpu.prefetch_layers(step, list(range(1, cfg.sources)))
            for layer in range(len(gpu.layers)):
                gpu.gather_layer(step, layer, stream=g)
                ev = torch.cuda.Event()
                ev.record(g)
                main.wait_event(ev)  # the layer's consumer after its gather
                filler.add_(1)
            res = orc.step(step)
            torch.cuda.synchronize()
            assert gpu.status() == (0, 0)
            loc = _as_u32(gpu.loc)
            for r in range(cfg.requests):
                assert np.array_equal(loc[r], res[r]["loc"]), (step, r)
                stg = gpu.staging[r].cpu().view(torch.int16).numpy().view(np.uint16)
                assert np.array_equal(stg, res[r]["staging"]), (step, r)
    finally:
        gpu.close()
        orc.pool.close()


def test_union_staging_failures():
    # an out-of-range row and budget overflows: empty union lists
    cfg = TINY.scaled(name="ubudget", tag=50, requests=2, sources=1, hot=16, topk=64,
                      queries=2, verify_core=32, residency=0.0, steps=4)
    compare_run(cfg, union=True, gather_impl=1)
    cfg = TINY.scaled(name="urange", tag=46, requests=2, sources=2, steps=4, residency=0.6)
    compare_run(cfg, union=True, gather_impl=1, patch=_bad_row)


def _bad_row(wl):
    """Step 3 of request 1 source 0 selects row L (one past the end)."""
    sel = wl.selections()
    sel[2, 1, 0, 0, 5] = wl.length(1, 3)


@pytest.mark.parametrize("mode", ["fused-vec", "fused-tma", "split-vec", "split-tma",
                                  "fused-tma-late"])
def test_out_of_range_row_keeps_only_step1_rows(mode):
    """The failed item's step-1 rows are gathered, every other entry is zeros."""
    cfg = TINY.scaled(name="range", tag=46, requests=2, sources=2, steps=4, residency=0.6)
    compare_run(cfg, fused=mode.startswith("fused"), gather_impl=IMPLS[mode.split("-")[1]],
                patch=_bad_row, early=0 if mode.endswith("late") else 1)


@pytest.mark.parametrize("mode", ["fused-vec", "fused-tma", "split-tma", "fused-tma-late"])
def test_budget_overflow_keeps_only_step1_rows(mode):
    # 16 hot slots, 40 % residency: most steps need more victims than slots,
    # and their items still hold step-1 rows
    cfg = TINY.scaled(name="budget", tag=47, requests=2, sources=1, hot=16, topk=64,
                      residency=0.4, steps=4)
    compare_run(cfg, fused=mode.startswith("fused"), gather_impl=IMPLS[mode.split("-")[1]],
                early=0 if mode.endswith("late") else 1)


# ------------------------------------------------------------ full size

@pytest.mark.parametrize("impl,early", [(0, 1), (1, 1), (1, 0)])
def test_c8_full_size_sampled(impl, early):
    compare_run(C8, sampled=[0, 5], gather_impl=impl, early=early)


def test_c64_full_size_sampled():
    compare_run(C64, sampled=[0, 63])


def test_c64_union_full_size_sampled():
    compare_run(C64, sampled=[0, 63], union=True)


def test_decode_step_fallback_matches_split_calls():
    """dhs_decode_step where some appending pairs are not resolved in the
    step (it must append separately) gives what dhs_append + dhs_resolve +
    dhs_gather give."""
    import ctypes
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    cfg = TINY.scaled(name="fallback", tag=48, requests=3, sources=2, steps=3,
                      residency=0.3, hot=300)
    wl = Workload(cfg)
    a, b = GpuRun(cfg, wl), GpuRun(cfg, wl)
    try:
        for step in range(1, cfg.total_steps + 1):
            apps, n = a._appends[step - 1]
            st, items = a._steps[step - 1]
            sub = [items[i] for i in range(len(items)) if items[i].req == 1]
            st_a, keep_a = dhs.make_step(step, sub)
            assert dhs.lib.dhs_append(a.pool.h, apps, n) == 0
            assert dhs.lib.dhs_resolve(a.pool.h, ctypes.byref(st_a)) == 0
            assert dhs.lib.dhs_gather(a.pool.h, ctypes.byref(st_a)) == 0
            apps_b, nb = b._appends[step - 1]
            st_b0, items_b = b._steps[step - 1]
            sub_b = [items_b[i] for i in range(len(items_b)) if items_b[i].req == 1]
            st_b, keep_b = dhs.make_step(step, sub_b)
            assert dhs.lib.dhs_decode_step(b.pool.h, apps_b, nb, ctypes.byref(st_b)) == 0
            torch.cuda.synchronize()
            assert a.status() == (0, 0) and b.status() == (0, 0)
            assert torch.equal(a.loc[1], b.loc[1]) and torch.equal(a.counters[1], b.counters[1])
            assert torch.equal(a.staging[1].view(torch.int16), b.staging[1].view(torch.int16))
        for r in range(cfg.requests):
            for s in range(cfg.sources):
                L = wl.length(r, cfg.total_steps)
                assert np.array_equal(a.host_rows(r, s, 0, L), b.host_rows(r, s, 0, L))
                assert a.pool.read_state(r, s)[3][1] == b.pool.read_state(r, s)[3][1] == L
    finally:
        a.close()
        b.close()


def test_c128_full_size_sampled():
    # request 0 is reclaimed (no optional pages), request 127 stays resident
    compare_run(C128, sampled=[0, 127])


def test_long_full_size_sampled():
    compare_run(LONG, sampled=[0, 31])


def test_admission_rejects_misaligned_host_rows():
    """Rows move between HBM and the host copy in 16-byte chunks: a host
    copy that is not 16-byte aligned is refused, for both admissions."""
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    pool = dhs.Pool(max_requests=2, sources=1, row_bytes=16, page_rows=4, tail_rows=2,
                    hot_rows=4, max_queries=1, max_topk=4, max_rows_per_request=16,
                    optional_pages=4)
    host = dhs.HostRows(4096)
    dev = torch.zeros(16 * 8, dtype=torch.int16, device="cuda")
    try:
        rc, _ = pool.admit(0, 0, host.ptr + 8, 8, None)
        assert rc == dhs.DHS_EINVAL
        rc, _ = pool.admit_device(0, 0, dev.data_ptr(), host.ptr + 8, 8, None)
        assert rc == dhs.DHS_EINVAL
        rc, _ = pool.admit_device(0, 0, dev.data_ptr(), host.ptr, 8, None)
        assert rc == 0
        torch.cuda.synchronize()
    finally:
        pool.close()
        host.close()


def test_decode_step_host_matches_device_path():
    """dhs_decode_step_host (host selections and decode rows in, host
    locations and counters out, one call) gives what the device-side
    dhs_decode_step leaves in device memory."""
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    cfg = SMALL[1]  # verify block of 3 queries, ragged k, appends of 1-4 rows
    wl = Workload(cfg)
    a, b = GpuRun(cfg, wl), GpuRun(cfg, wl)
    try:
        loc_h = torch.empty(b.loc.shape, dtype=b.loc.dtype).pin_memory()
        cnt_h = torch.empty(b.counters.shape, dtype=b.counters.dtype).pin_memory()
        for step in range(1, cfg.total_steps + 1):
            sel_h = b.sel[step - 1].cpu().pin_memory()
            rows_h = b.app_rows[step - 1].cpu().pin_memory()
            b.sel[step - 1].zero_()  # the call must bring the inputs in itself
            b.app_rows[step - 1].zero_()
            a.step(step)

            def span(dst, src):
                return (dst.data_ptr(), src.data_ptr(), src.numel() * src.element_size())

            b.step_host(step, [span(b.sel[step - 1], sel_h), span(b.app_rows[step - 1], rows_h)],
                        [span(loc_h, b.loc), span(cnt_h, b.counters)])
            torch.cuda.synchronize()
            assert torch.equal(loc_h, a.loc.cpu()) and torch.equal(cnt_h, a.counters.cpu())
            assert torch.equal(a.staging.view(torch.int16), b.staging.view(torch.int16))
        assert a.status() == (0, 0) and b.status() == (0, 0)
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("streams", [False, True])
def test_decode_step_host_async_pipelined_matches_device_path(streams):
    """dhs_decode_step_host_async with later steps enqueued before step s's
    outputs are read (two host output sets; with `streams`, four, the input
    and output copies on their own streams and four device output blocks,
    as the bench's e2e runs it) gives what the device-side dhs_decode_step
    leaves in device memory, step by step."""
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    cfg = SMALL[1]
    wl = Workload(cfg)
    a, b = GpuRun(cfg, wl), GpuRun(cfg, wl)
    try:
        def span(dst, src):
            return (dst.data_ptr(), src.data_ptr(), src.numel() * src.element_size())

        # host output sets; step s's outputs are read after step s+D-1 is
        # enqueued.  Without streams every copy is on the pool's stream, which
        # orders the one device output block's reuse.
        D = 4 if streams else 2
        blocks = [b.output_block(i if streams else 0) for i in range(D)]
        cnt_off = b.counters.data_ptr() - b.step_out.data_ptr()
        loc_n, cnt_n = b.loc.numel() * 4, b.counters.numel() * 4
        outs = [torch.empty(blk.shape, dtype=torch.uint8).pin_memory() for blk in blocks]
        ins = [b.step_in[s].cpu().pin_memory() for s in range(cfg.total_steps)]
        b.step_in.zero_()  # the calls must bring the inputs in themselves
        want = []
        for step in range(1, cfg.total_steps + 1):
            a.step(step)
            want.append((a.loc.cpu(), a.counters.cpu(), a.staging.clone()))
        pool_stream = torch.cuda.current_stream()
        s_in = torch.cuda.Stream() if streams else None
        s_out = torch.cuda.Stream() if streams else None
        out_done = [torch.cuda.Event() for _ in range(D)]

        def check(j, step):
            o = outs[j]
            loc_w, cnt_w, _ = want[step - 1]
            assert torch.equal(o[:loc_n].view(torch.int32).view(loc_w.shape), loc_w), step
            assert torch.equal(o[cnt_off:cnt_off + cnt_n].view(torch.int32).view(cnt_w.shape),
                               cnt_w), step

        T = cfg.total_steps
        for step in range(1, T + 1):
            j = (step - 1) % D  # set j's last outputs (step - D) are already read
            io = b.host_io(step, [span(b.step_in[step - 1], ins[step - 1])],
                           [span(outs[j], blocks[j])], out_set=j if streams else 0)
            b.step_host(step, io=io, wait=False, in_stream=s_in, out_stream=s_out)
            out_done[j].record(s_out if streams else pool_stream)
            if step >= D:
                r = step - (D - 1)
                out_done[(r - 1) % D].synchronize()
                check((r - 1) % D, r)
        for r in range(max(1, T - D + 2), T + 1):
            out_done[(r - 1) % D].synchronize()
            check((r - 1) % D, r)
        torch.cuda.synchronize()
        assert torch.equal(want[-1][2].view(torch.int16), b.staging.view(torch.int16))
        assert a.status() == (0, 0) and b.status() == (0, 0)
    finally:
        a.close()
        b.close()


def test_degenerate_steps():
    """Through the C ABI: an empty step (no items, no appends) changes
    nothing in any entry point; an item with k = 0 resolves nothing (zero
    counters); steps of gather-only items gather without resolving, fused or
    not; ordinary steps around them still match the oracle."""
    import ctypes
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    from oracle.run import OracleRun
    cfg = TINY.scaled(name="degen", tag=56, requests=2, sources=1, steps=3, residency=0.5)
    wl = Workload(cfg)
    gpu, orc = GpuRun(cfg, wl), OracleRun(cfg, wl)
    h = gpu.pool.h

    def check(step):
        res = orc.step(step)
        for r in range(cfg.requests):
            assert np.array_equal(gpu.loc[r].cpu().numpy().view(np.uint32), res[r]["loc"])
            assert np.array_equal(gpu.counters[r].cpu().numpy().view(np.uint32),
                                  res[r]["counters"])
            stg = gpu.staging[r].cpu().view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(stg, res[r]["staging"])

    try:
        empty, _keep = dhs.make_step(1, [])
        for fn in (dhs.lib.dhs_resolve, dhs.lib.dhs_gather, dhs.lib.dhs_resolve_gather):
            assert fn(h, ctypes.byref(empty)) == 0
        assert dhs.lib.dhs_decode_step(h, None, 0, ctypes.byref(empty)) == 0
        # k = 0
        cnt = torch.full((8,), 7, dtype=torch.int32, device="cuda")
        it = dhs.dhs_item()
        it.req, it.src, it.queries, it.topk = 0, 0, 1, 0
        it.sel_dev, it.loc_dev = gpu.sel[0, 0, 0].data_ptr(), gpu.loc[0, 0].data_ptr()
        it.counters_dev, it.staging_dev = cnt.data_ptr(), gpu.staging[0, 0].data_ptr()
        st0, _keep0 = dhs.make_step(1, [it])
        assert dhs.lib.dhs_resolve_gather(h, ctypes.byref(st0)) == 0
        torch.cuda.synchronize()
        assert gpu.status() == (0, 0) and not cnt.cpu().any()
        gpu.step(1)
        check(1)
        # gather-only items on step 1's locations, into other staging
        other = torch.zeros_like(gpu.staging)
        items = []
        for r in range(cfg.requests):
            g = dhs.dhs_item()
            g.req, g.src, g.queries, g.topk = r, 0, cfg.queries, cfg.topk
            g.flags = dhs.DHS_ITEM_GATHER_ONLY
            g.loc_dev, g.staging_dev = gpu.loc[r, 0].data_ptr(), other[r, 0].data_ptr()
            items.append(g)
        stg, _keepg = dhs.make_step(1, items)
        for fn in (dhs.lib.dhs_gather, dhs.lib.dhs_resolve_gather):
            other.zero_()
            assert fn(h, ctypes.byref(stg)) == 0
            torch.cuda.synchronize()
            assert torch.equal(other.view(torch.int16), gpu.staging.view(torch.int16))
        for step in (2, 3):
            gpu.step(step)
            check(step)
        assert gpu.status() == (0, 0)
    finally:
        gpu.close()
        orc.pool.close()


# 400 (request, source) pairs: two resolve and copy launches (at most 256
# items each) and two gather launches (at most 384 items each) per step
MANY = TINY.scaled(name="many", tag=57, requests=200, sources=2, history=512, tail=16,
                   hot=96, topk=48, steps=4, residency=0.3)


@pytest.mark.parametrize("mode", ["fused-tma", "split-vec", "fused-tma-union"])
def test_steps_of_several_launches_per_kernel(mode):
    compare_run(MANY, fused=mode.startswith("fused"), gather_impl=IMPLS[mode.split("-")[1]],
                union=mode.endswith("union"))


@pytest.mark.parametrize("mode", ["fused-tma", "split-vec", "fused-tma-union", "fused-tma-late-copy"])
def test_resolve_two_ctas_per_sm(mode):
    """Resolve launches of more than 32 items as 512-thread CTAs two per SM
    (what the pool picks when the host copy waits for the resolve grid):
    bit-exact on steps of 400 pairs, fused and split, both layouts, with the
    copy overlapped and launched after the resolve grid."""
    compare_run(MANY, fused=mode.startswith("fused"), gather_impl=IMPLS[mode.split("-")[1]],
                union=mode.endswith("union"), resolve_paired=1,
                copy_pdl=0 if mode.endswith("late-copy") else None)


MAXHOT = TINY.scaled(name="maxhot", tag=53, requests=1, sources=1, hot=16384, history=65536,
                     topk=4096, residency=0.0, steps=10, window=4096, frac_recent=0.3,
                     zipf_s=0.6, row_elems=64)


@pytest.mark.parametrize("mode", ["fused-tma", "split-vec", "fused-tma-union"])
def test_largest_hot_cache_fills_and_evicts(mode):
    """B at its maximum (16384 slots): about 4000 misses a step fill the hot
    cache by step 5, and from step 6 every step evicts ~1900 rows."""
    compare_run(MAXHOT, fused=mode.startswith("fused"), gather_impl=IMPLS[mode.split("-")[1]],
                union=mode.endswith("union"))


def test_large_rows_take_the_tma_gather_with_opt_in_shared_memory():
    """4 KB rows: a 16-entry TMA tile needs 64 KB of shared memory (past the
    48 KB default), which the pool opts in to; bit-exact in every mode."""
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    cfg = TINY.scaled(name="rows4k", tag=52, row_elems=2048, history=1024, tail=16,
                      hot=128, topk=64, steps=4, requests=2)
    gpu = GpuRun(cfg, Workload(cfg))
    try:
        assert gpu.pool.get_option(dhs.DHS_OPT_GATHER_IMPL) == 1
    finally:
        gpu.close()
    compare_run(cfg, gather_impl=1)
    compare_run(cfg, gather_impl=1, fused=False)


def test_rows_too_large_for_a_tma_tile_use_the_vector_gather():
    """16 KB rows: a 16-entry tile of them does not fit in a block's shared memory, so the
    pool refuses the TMA gather and runs the vector gather, bit-exact."""
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    cfg = TINY.scaled(name="bigrows", tag=51, row_elems=8192, history=1024, tail=16,
                      hot=128, topk=64, steps=4, requests=2)
    gpu = GpuRun(cfg, Workload(cfg))
    try:
        assert gpu.pool.get_option(dhs.DHS_OPT_GATHER_IMPL) == 0
        with pytest.raises(Exception):
            gpu.pool.set_option(dhs.DHS_OPT_GATHER_IMPL, 1)
    finally:
        gpu.close()
    compare_run(cfg, gather_impl=0)
    compare_run(cfg, gather_impl=0, fused=False)

"""Pins of the CPU oracle against facts that do not come from the oracle.

  * hand-worked traces (tests/golden), including EBUDGET roll-back, ERANGE,
    verify-block unions, ring wrap, incomplete pages, admission/reclaim;
  * LRU closed forms: with one hot-candidate row per step a row hits iff its
    LRU stack distance (Mattson et al., 1970) is below B, and the cache holds
    exactly the B most recently used rows; with batched steps, rows used at
    step t stay cached while at most B distinct rows are used from t on;
  * special cases with closed-form counts (all history resident; repeated
    selection; B larger than every row ever selected);
  * library routines (numpy unique) for the union size;
  * byte truth: every gathered row equals the generator's payload of the
    selected row, host rows after appends equal the payload.

Sources: "Adaptive DHiSparse: Speculative Decoding over a Load-Adaptive KV
Hierarchy", How it works (Memory split, Reclamation and refill, Resolution,
Speculative state, Model-specific reuse) and Limits.
"""
import numpy as np
import pytest

import dhs_workload
from dhs_workload.configs import TINY, Config, Workload
from fixture_runner import OracleAdapter, run_trace

import oracle
from oracle import OraclePool, decode
from oracle.run import OracleRun

TRACES = ["resolve_micro_b2.txt", "resolve_micro_b3_pairs.txt",
          "admission_micro.txt", "backup_refill_micro.txt", "window_micro.txt",
          "resolve_micro_same_step.txt"]


@pytest.mark.parametrize("trace", TRACES)
def test_golden_trace(oracle_lib, gen_lib, trace):
    run_trace(trace, OracleAdapter())


# ------------------------------------------------------------ LRU closed forms

def _hot_only_pool(B, N=4096, T=1, E=8):
    p = OraclePool(1, 1, T, B, E, 64, N + 64, 0)
    none = np.zeros(N // 64, np.uint8)  # no optional pages
    assert p.admit(0, 0, N, none, None) == (0, 0)
    return p


@pytest.mark.parametrize("B", [1, 2, 4, 7])
def test_mattson_stack_distance(oracle_lib, B):
    """One row per step, no tail/optional hits: hit iff fewer than B distinct
    other rows were used since the row's previous use (LRU stack distance),
    and the cache holds the min(B, distinct) most recently used rows."""
    rng = np.random.default_rng(B)
    p = _hot_only_pool(B)
    trace = rng.integers(0, 3 * B + 2, size=400)
    history = []
    for step, row in enumerate(trace, 1):
        row = int(row)
        if row in history:
            last = len(history) - 1 - history[::-1].index(row)
            distance = len(set(history[last + 1:]))
            expect_hit = distance < B
        else:
            expect_hit = False
        rc, loc, cnt = p.resolve(step, 0, 0, np.array([[row]], np.int32))
        assert rc == 0
        assert cnt[4] == (1 if expect_hit else 0), (step, row)
        assert cnt[5] == (0 if expect_hit else 1), (step, row)
        history.append(row)
        mru = []
        for x in reversed(history):
            if x not in mru:
                mru.append(x)
        tags, stamps, _, _ = p.state(0, 0)
        assert set(int(t) for t in tags if t >= 0) == set(mru[:B])


@pytest.mark.parametrize("seed", range(6))
def test_lru_keeps_recent_working_set(oracle_lib, seed):
    """Batched steps: after step v, if the rows used in steps t..v number at
    most B, all of them are still cached.  (Evicting a row last used at or
    after t needs all B slots to hold such rows plus one more new row.)"""
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(2, 9))
    p = _hot_only_pool(B)
    used = []
    for step in range(1, 80):
        k = int(rng.integers(1, B + 1))
        sel = np.sort(rng.choice(3 * B, size=k, replace=False)).astype(np.int32)
        rc, loc, cnt = p.resolve(step, 0, 0, sel[None])
        assert rc == 0
        used.append(set(sel.tolist()))
        tags = {int(x) for x in p.state(0, 0)[0] if x >= 0}
        window = set()
        for t in range(len(used) - 1, -1, -1):
            window |= used[t]
            if len(window) > B:
                break
            assert window <= tags, (step, t)


def test_closed_form_all_resident(oracle_lib):
    """Every complete page resident, decode rows still in the tail: every
    selected row resolves in step 1 (tail rows >= L-T, the rest optional)."""
    N, T, B, k = 512, 32, 16, 40
    p = OraclePool(1, 1, T, B, 8, 64, N + 64, N // 64)
    assert p.admit(0, 0, N, None, None) == (0, 0)
    rng = np.random.default_rng(7)
    L = N
    for step in range(1, 20):
        assert p.append(0, 0, 1) == 0
        L += 1
        sel = rng.choice(L, size=k, replace=False).astype(np.int32)
        rc, loc, cnt = p.resolve(step, 0, 0, sel[None])
        assert rc == 0
        n_tail = int((sel >= L - T).sum())
        assert list(cnt) == [k, k, n_tail, k - n_tail, 0, 0, 0, 0]


def test_closed_form_repeated_selection(oracle_lib):
    """No residency, no appends, the same k <= B rows each step: step 1 fetches
    every non-tail row from host; every later step hits all of them."""
    N, T, B, k = 1000, 8, 64, 50
    p = OraclePool(1, 1, T, B, 8, 64, N + 8, 0)
    assert p.admit(0, 0, N, np.zeros(N // 64, np.uint8), None) == (0, 0)
    rng = np.random.default_rng(3)
    sel = rng.choice(N, size=k, replace=False).astype(np.int32)
    n_tail = int((sel >= N - T).sum())
    for step in range(1, 6):
        rc, loc, cnt = p.resolve(step, 0, 0, sel[None])
        assert rc == 0
        hot, host = (0, k - n_tail) if step == 1 else (k - n_tail, 0)
        assert list(cnt[:6]) == [k, k, n_tail, 0, hot, host]
        assert cnt[7] == 0


def test_closed_form_no_eviction(oracle_lib):
    """B >= every row ever selected: no evictions, and the host fetches over
    the run equal the distinct rows that step 1 never resolves."""
    N, T, B = 300, 4, 400
    p = OraclePool(1, 1, T, B, 8, 64, N + 8, 0)
    assert p.admit(0, 0, N, np.zeros(N // 64, np.uint8), None) == (0, 0)
    rng = np.random.default_rng(5)
    seen, host = set(), 0
    for step in range(1, 30):
        sel = rng.integers(0, N, size=(2, 17)).astype(np.int32)
        rc, loc, cnt = p.resolve(step, 0, 0, sel)
        assert rc == 0 and cnt[7] == 0
        host += int(cnt[5])
        seen |= {int(x) for x in sel.ravel() if x < N - T}
    assert host == len(seen)


def test_union_size_matches_numpy_unique(oracle_lib):
    p = _hot_only_pool(64)
    rng = np.random.default_rng(11)
    for step in range(1, 20):
        sel = rng.integers(0, 80, size=(3, 9)).astype(np.int32)
        rc, loc, cnt = p.resolve(step, 0, 0, sel)
        assert rc == 0
        assert cnt[0] == sel.size and cnt[1] == len(np.unique(sel))
        # duplicates share one location
        flat, lf = sel.ravel(), loc.ravel()
        for v in np.unique(flat):
            assert len(set(lf[flat == v].tolist())) == 1


def test_range_and_tail_boundary(oracle_lib):
    N, T, B = 256, 16, 8
    p = OraclePool(1, 1, T, B, 8, 64, N + 8, 8)
    p.admit(0, 0, N, np.array([0, 0, 0, 1], np.uint8), None)  # page 3 resident
    for bad in ([[N]], [[-1]], [[0, N + 3]]):
        rc, loc, cnt = p.resolve(1, 0, 0, np.array(bad, np.int32))
        assert rc == "erange" and (loc == oracle.NO_LOC).all() and not cnt.any()
    # a failed step still locates what step 1 holds: the tail row and the row
    # on resident page 3, not row 0 (page 0 absent) nor the out-of-range row
    rc, loc, cnt = p.resolve(1, 0, 0, np.array([[N - 1, N, 3 * 64 + 5, 0]], np.int32))
    assert rc == "erange" and not cnt.any()
    tier, idx = decode(loc.ravel()[[0, 2]])
    assert tier.tolist() == [0, 1] and idx.tolist() == [(N - 1) % T, 0 * 64 + 5]
    assert (loc.ravel()[[1, 3]] == oracle.NO_LOC).all()
    # row L-T is tail; L-T-1 lies in resident page 3 -> optional
    rc, loc, cnt = p.resolve(1, 0, 0, np.array([[N - T, N - T - 1, N - 1]], np.int32))
    assert rc == 0
    tier, idx = decode(loc.ravel())
    assert tier.tolist() == [0, 1, 0]
    assert idx.tolist() == [(N - T) % T, 0 * 64 + (N - T - 1) % 64, (N - 1) % T]


def test_admission_capacity_rule(oracle_lib):
    """required + optional + reserve <= capacity, checked on optional pages."""
    p = OraclePool(2, 1, 4, 4, 8, 64, 1024, capacity=10, reserve=2)
    assert p.admit(0, 0, 64 * 5, None, None) == (0, 0)
    assert p.admit(1, 0, 64 * 4, None, None) == ("wouldwait", 1)
    assert p.admit(1, 0, 64 * 3 + 10, None, None) == (0, 0)
    assert p.used() == 8
    assert p.admit(1, 0, 64, None, None)[0] == "estate"


# ------------------------------------------------------------ whole workload

def _tiny_scaled(**kw):
    return TINY.scaled(**kw)


@pytest.mark.parametrize("cfg", [
    TINY,
    _tiny_scaled(name="tiny_q3", tag=31, queries=3, verify_core=200, hot=1024,
                 steps=8, append_lo=1, append_hi=3),
    _tiny_scaled(name="tiny_reuse", tag=32, sources=3, requests=2,
                 reuse_layers=2, shared_selection=True, steps=6, residency=0.2),
])
def test_workload_byte_truth_and_invariants(oracle_lib, gen_lib, cfg):
    run = OracleRun(cfg)
    wl = run.wl
    for step in range(1, cfg.total_steps + 1):
        res = run.step(step)
        for r, out in res.items():
            L = wl.length(r, step)
            for s in range(cfg.sources):
                assert out["rc"][s] == 0
                cnt = out["counters"][s]
                sel = wl.sel(step, r, s)
                assert cnt[0] == sel.size and cnt[1] == len(np.unique(sel))
                assert cnt[2] + cnt[3] + cnt[4] + cnt[5] == cnt[1]
                assert cnt[6] <= cfg.hot
                if cnt[5]:
                    assert cnt[6] == cfg.hot
                assert run.pool.check(r, s) == 0
                tier, _ = decode(out["loc"][s].ravel())
                rows = sel.ravel()
                # rows generated during decoding never resolve as optional
                assert not ((tier == oracle.TIER_OPT) & (rows >= cfg.history)).any()
                # tail rows are exactly [L-T, L)
                assert np.array_equal(tier == oracle.TIER_TAIL, rows >= L - cfg.tail)
            for layer, (kind, s) in enumerate(run.layers()):
                sel = wl.sel(step, r, s).ravel()
                st = out["staging"][layer].reshape(-1, cfg.row_elems)
                for e in range(0, sel.size, max(1, sel.size // 97)):
                    want = dhs_workload.payload_row(cfg.tag, s, r, int(sel[e]),
                                                    cfg.row_elems)
                    assert np.array_equal(st[e], want), (step, r, layer, e)
            for layer, (kind, s) in enumerate(run.layers()):
                if kind == "reuse":  # Reuse layers inherit source 0's locations
                    assert np.array_equal(out["staging"][layer], out["staging"][0])
    # the host copy holds every row: imported and written-through decode rows
    for r in run.requests:
        for s in range(cfg.sources):
            L = wl.length(r, cfg.total_steps)
            got = run.pool.rows(r, s, 0, 0, L)
            want = dhs_workload.payload_rows(cfg.tag, s, r, 0, L, cfg.row_elems)
            assert np.array_equal(got, want)


# ------------------------------------------------------------ window sources

@pytest.mark.parametrize("T", [1, 5, 16])
def test_window_source_closed_form(oracle_lib, gen_lib, T):
    """A window source ("Speculative state": a drafter retains only the rows
    its window covers, stored as a ring) beside an ordinary one, under random
    appends and selections.  Closed form: a selection inside [L-T, L)
    resolves entirely from the ring -- entry e at tail index pair*T +
    sel[e] mod T, counters (Q*k, distinct, distinct, 0, 0, 0, 0, 0) -- and
    gathers the payload of its rows; a selection with any row outside it is
    ERANGE, its in-window entries keeping their ring locations and the rest
    none.  The hot cache is never touched and no capacity is taken."""
    rng = np.random.default_rng(T)
    E, tag = 8, 96
    p = OraclePool(2, 2, T, 4, E, 4, 400, 16)
    assert p.admit(0, 0, 40, None, dhs_workload.payload_rows(tag, 0, 0, 0, 40, E))[0] == 0
    used = p.used()
    N = int(rng.integers(0, 60))
    m = min(N, T)
    assert p.admit_window(1, 1, N, dhs_workload.payload_rows(tag, 1, 1, N - m, m, E)) == 0
    assert p.used() == used
    pair, L = 1 * 2 + 1, N
    for step in range(1, 60):
        a = int(rng.integers(0, T + 1))
        if a and L + a <= 400:
            assert p.append(1, 1, a, dhs_workload.payload_rows(tag, 1, 1, L, a, E)) == 0
            L += a
        lo = max(0, L - T)
        Q, k = int(rng.integers(1, 4)), int(rng.integers(1, 9))
        if L == 0 or rng.random() < 0.3:  # some rows outside the window
            sel = rng.integers(-2, L + 3, size=(Q, k))
        else:
            sel = rng.integers(lo, L, size=(Q, k))
        rc, loc, cnt = p.resolve(step, 1, 1, sel)
        inside = (sel >= lo) & (sel < L)
        want_loc = np.where(inside, pair * T + np.mod(sel, T), 0xFFFFFFFF).astype(np.uint32)
        assert np.array_equal(loc, want_loc), (step, sel, loc)
        if inside.all():
            u = np.unique(sel).size
            assert rc == 0 and list(cnt) == [Q * k, u, u, 0, 0, 0, 0, 0]
            rcg, st = p.gather(loc)
            assert rcg == 0
            for q in range(Q):
                for i in range(k):
                    want = dhs_workload.payload_row(tag, 1, 1, int(sel[q, i]), E)
                    assert np.array_equal(st[q, i], want), (step, q, i)
        else:
            assert rc == "erange" and not cnt.any()
        tags, stamps, pages, lens = p.state(1, 1)
        assert (tags == -1).all() and (stamps == 0).all() and (pages == -1).all()
        assert lens == (0, L, 1)
        assert p.check(1, 1) == 0
    p.close()

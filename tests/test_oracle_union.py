"""Pins of the oracle's union staging layout (each distinct row of a verify
block staged once, plus per-query index lists).

The layout is pinned against things outside the oracle: numpy's sorted
unique of the selection (the union and each entry's rank in it), the
generator's payload of every union row (byte truth), and the oracle's own
per-query layout through the identity loc[q][i] == union_loc[index[q][i]]
(the per-query layout is pinned by the other oracle tests)."""
import numpy as np
import pytest

import dhs_workload
import oracle
from dhs_workload.configs import TINY
from oracle import OraclePool
from oracle.run import OracleRun

CFGS = [
    TINY.scaled(name="u_q3", tag=61, queries=3, verify_core=60, topk=90, hot=400,
                steps=8, append_lo=1, append_hi=3, requests=2, sources=2),
    TINY.scaled(name="u_q8_evict", tag=62, queries=8, verify_core=40, topk=50,
                hot=300, residency=0.0, steps=6, requests=1, sources=1),
    TINY.scaled(name="u_reuse", tag=63, requests=2, sources=2, reuse_layers=2,
                shared_selection=True, residency=0.3, steps=5),
]


@pytest.mark.parametrize("cfg", CFGS, ids=[c.name for c in CFGS])
def test_union_layout(oracle_lib, gen_lib, cfg):
    uni = OracleRun(cfg, union=True)
    per = OracleRun(cfg, wl=uni.wl)
    wl = uni.wl
    for step in range(1, cfg.total_steps + 1):
        ru, rp = uni.step(step), per.step(step)
        for r in uni.requests:
            u, p = ru[r], rp[r]
            assert u["rc"] == p["rc"]
            assert np.array_equal(u["counters"], p["counters"])
            for s in range(cfg.sources):
                sel = wl.sel(step, r, s).ravel()
                rows = np.unique(sel)
                U = int(u["counters"][s][1])
                assert U == rows.size
                idx = u["index"][s].ravel()
                loc = u["loc"][s]
                assert np.array_equal(idx, np.searchsorted(rows, sel))
                assert (loc[U:] == oracle.END_LOC).all()
                assert np.array_equal(loc[idx], p["loc"][s].ravel())
            for layer, (kind, s) in enumerate(uni.layers()):
                rows = np.unique(wl.sel(step, r, s))
                st = u["staging"][layer]
                assert st.shape == (rows.size, cfg.row_elems)
                for j in range(0, rows.size, max(1, rows.size // 37)):
                    want = dhs_workload.payload_row(cfg.tag, s, r, int(rows[j]),
                                                    cfg.row_elems)
                    assert np.array_equal(st[j], want), (step, r, layer, j)
                idx = u["index"][s].reshape(-1)
                pq = p["staging"][layer].reshape(-1, cfg.row_elems)
                assert np.array_equal(st[idx], pq)
    uni.pool.close()
    per.pool.close()


def test_union_error_leaves_empty_list(oracle_lib):
    N, T, B = 256, 16, 8
    p = OraclePool(1, 1, T, B, 8, 64, N + 8, 8)
    p.admit(0, 0, N, None, None)
    rc, loc, idx, cnt = p.resolve_union(1, 0, 0, np.array([[3, N], [4, 5]], np.int32))
    assert rc == "erange"
    assert (loc == oracle.END_LOC).all() and (idx == -1).all() and not cnt.any()
    # budget overflow: 3 distinct misses, 2 hot slots
    p2 = OraclePool(1, 1, 1, 2, 8, 64, N + 8, 0)
    assert p2.admit(0, 0, N, np.zeros(N // 64, np.uint8), None)[0] == 0
    rc, loc, idx, cnt = p2.resolve_union(1, 0, 0, np.array([[1, 2], [2, 3]], np.int32))
    assert rc == "ebudget"
    assert (loc == oracle.END_LOC).all() and (idx == -1).all()
    tags, stamps, _, _ = p2.state(0, 0)
    assert (tags == -1).all() and (stamps == 0).all()
    # a following step that fits works and lays out the union
    rc, loc, idx, cnt = p2.resolve_union(2, 0, 0, np.array([[9, 7], [7, 9]], np.int32))
    assert rc == 0 and cnt[1] == 2 and idx.tolist() == [[1, 0], [0, 1]]
    assert loc[2:].tolist() == [oracle.END_LOC] * 2


def test_verify_block_fetches_each_missing_row_once(oracle_lib):
    """A verify block's queries fetch each missing row once between them
    ("Adaptive DHiSparse", How it works / Speculative state).  From the pool's state
    before each step (tail window, ready pages, hot tags), the rows no tier
    holds are the block's distinct selected rows minus those: the host
    fetches must equal their count -- once per row however many queries
    select it -- which is at most the sum of each query's own missing rows."""
    rng = np.random.default_rng(5)
    R, S, T, B, E, PR, N = 1, 1, 8, 48, 4, 16, 512
    p = OraclePool(R, S, T, B, E, PR, N + 64, 40)
    mask = (rng.random(N // PR) < 0.4).astype(np.uint8)
    assert p.admit(0, 0, N, mask, None)[0] == 0
    L, shared = N, 0
    for step in range(1, 25):
        assert p.append(0, 0, 1) == 0
        L += 1
        core = rng.choice(L, size=12, replace=False)
        sel = np.stack([np.concatenate([core, rng.choice(L, size=4, replace=False)])
                        for _ in range(3)]).astype(np.int32)
        tags, _, page_slot, _ = p.state(0, 0)
        held = set(tags[tags >= 0].tolist())

        def missing(rows):
            out = set()
            for row in np.unique(rows).tolist():
                if row >= L - T:
                    continue  # tail
                if (row // PR + 1) * PR <= N and page_slot[row // PR] >= 0:
                    continue  # ready optional page
                if row not in held:
                    out.add(row)
            return out

        want = missing(sel)
        per_query = sum(len(missing(q)) for q in sel)
        rc, loc, cnt = p.resolve(step, 0, 0, sel)
        if rc != 0:
            continue
        assert int(cnt[5]) == len(want), (step, cnt, len(want))
        assert int(cnt[5]) <= per_query
        shared += per_query - int(cnt[5])
    assert shared > 0, "some missing rows must be selected by several queries"
    p.close()

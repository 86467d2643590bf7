"""The seeded input generators: bf16 rounding against torch's conversion,
payload statistics, selection shape (k distinct sorted rows, the recency /
Zipf mix, the verify-block overlap), exact residency counts, append ranges,
and determinism."""
import numpy as np
import pytest
import torch

import dhs_workload
from dhs_workload.configs import C64, CONFIGS, TINY, Config, Workload


def test_bf16_round_to_nearest_even_matches_torch(gen_lib):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, -2.5, 3.0e38, 1e-40, 65504.0,
                                  1.00390625, 1.01171875, 1.0078125],
                                 np.float32)])
    ours = dhs_workload.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_payload_is_standard_normal_and_deterministic(gen_lib):
    rows = dhs_workload.payload_rows(7, 0, 0, 0, 512, 576)
    vals = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert abs(vals.mean()) < 0.01 and abs(vals.std() - 1.0) < 0.01
    again = dhs_workload.payload_rows(7, 0, 0, 100, 10, 576)
    assert np.array_equal(again, rows[100:110])
    other = dhs_workload.payload_rows(7, 1, 0, 100, 10, 576)
    assert not np.array_equal(other, again)


def test_payload_pairs_layout(gen_lib):
    out = np.zeros((3, 20, 576), np.uint16)
    dhs_workload.payload_pairs_into(out.ctypes.data, 20, 9,
                                    [(0, 0), (1, 0), (0, 2)], 5, 12, 576, 0, 4)
    for i, (s, r) in enumerate([(0, 0), (1, 0), (0, 2)]):
        assert np.array_equal(out[i, :12], dhs_workload.payload_rows(9, s, r, 5, 12, 576))
        assert not out[i, 12:].any()


def test_selection_mix_and_shape(gen_lib):
    wl = Workload(TINY)
    c = TINY
    for step in (1, 5, 16):
        L = wl.length(0, step)
        sel = wl.sel(step, 0, 0)
        assert sel.shape == (1, c.topk)
        row = sel[0]
        assert (np.diff(row) > 0).all() and row[0] >= 0 and row[-1] < L
        W = min(c.window, L)
        in_window = ((row >= L - W) & (row < L)).sum()
        assert in_window >= min(round(0.7 * c.topk), W)


def test_verify_block_overlap(gen_lib):
    c = C64.scaled(requests=2, sources=1, steps=2, history=16384)
    wl = Workload(c)
    sel = wl.sel(1, 0, 0)
    assert sel.shape == (8, 2048)
    sets = [set(q.tolist()) for q in sel]
    for a in range(8):
        assert len(sets[a]) == 2048
        for b in range(a + 1, 8):
            assert len(sets[a] & sets[b]) == c.verify_core
    assert len(set().union(*sets)) == c.verify_core + 8 * (2048 - c.verify_core)


def test_residency_exact_counts(gen_lib):
    m = dhs_workload.residency(3, 1, 2, 512, 205)
    assert m.sum() == 205 and m.dtype == np.uint8
    assert np.array_equal(m, dhs_workload.residency(3, 1, 2, 512, 205))


def test_append_counts_range(gen_lib):
    a = dhs_workload.append_counts(3, 5, 1000, 1, 8)
    assert a.min() == 1 and a.max() == 8 and abs(a.mean() - 4.5) < 0.3


@pytest.mark.parametrize("name", list(CONFIGS))
def test_config_sizes(name):
    c = CONFIGS[name]
    assert c.max_rows >= c.history
    assert c.entries_per_step == c.requests * c.layers * c.queries * c.topk
    if name == "c8":
        assert c.entries_per_step == 65536
    if name == "long":
        assert c.entries_per_step == 393216 and c.resolved_per_step == 196608
    if name == "c128":
        assert c.pool_pages() == 61440


def test_temporal_locality_keeps_rows(gen_lib):
    c = TINY.scaled(rho=0.9, steps=4, tag=55)
    wl = Workload(c)
    a, b = set(wl.sel(2, 0, 0)[0].tolist()), set(wl.sel(3, 0, 0)[0].tolist())
    c0 = TINY.scaled(rho=0.0, steps=4, tag=55)
    wl0 = Workload(c0)
    a0, b0 = set(wl0.sel(2, 0, 0)[0].tolist()), set(wl0.sel(3, 0, 0)[0].tolist())
    assert len(a & b) > len(a0 & b0)

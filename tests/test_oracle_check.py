"""Pin of the oracle's invariant checker, orc_check.

orc_check states the invariants of one (request, source) that every correct
run keeps, so in every other test it only ever returns 0.  Here the oracle is
built with one extra test-only setter (tests/oracle_poke.c) that writes a
single field of the state; starting from a state that passes, each planted
violation must be reported by exactly the check that covers it:

  1  a hot tag outside [-1, L)             2  an empty slot with a stamp
  3  a filled slot with stamp 0            4  a tag held by two slots
  5  a ready page that is not complete     6  a ready page whose optional
                                              slot is not its own
  7  a page neither ready on the GPU nor backed up on the host
  8  a page both backed up and still pending backup
  9  a page counted as backed up whose host rows differ from the device's

Checks 7 and 9 are the pages' invariant that no row is without a copy, on
the GPU or on the host ("Adaptive DHiSparse", How it works / Reclamation and
refill; Resident-first admission defers the host backup, so a page can be
ready without one).  Checks 1-4 restate the hot cache of "Resolution" (B
slots, LRU stamps, empty slots tag -1 stamp 0); 5-6 restate "Memory split"
(only complete imported pages, one optional slot each).
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import dhs_workload
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
TAG = 97  # RNG key of these payloads
TAG_F, STAMP_F, PAGE_SLOT_F, BACKED_F, PEND_F, SLOT_PAIR_F, SLOT_PAGE_F, HOST_F = range(8)

R, S, T, B, E, PR, MAX_ROWS, CAP = 2, 1, 4, 4, 8, 4, 64, 16


@pytest.fixture(scope="module")
def poke_lib(tmp_path_factory):
    src = os.path.abspath(oracle.source_path())
    out = str(tmp_path_factory.mktemp("orc_poke") / "liborc_poke.so")
    subprocess.check_call(["gcc", "-O1", "-std=gnu11", "-fPIC", "-shared",
                           f'-DORC_SOURCE="{src}"', "-o", out,
                           os.path.join(HERE, "oracle_poke.c")])
    L = oracle.declare(ctypes.CDLL(out))
    L.orc_test_poke.restype = ctypes.c_int
    L.orc_test_poke.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int32, ctypes.c_int64, ctypes.c_int64]
    return L


@pytest.fixture
def pool(poke_lib, monkeypatch, gen_lib):
    """A valid two-request pool on the poke build of the oracle.

    Request 0 is admitted from device rows (18 rows: four complete pages and
    half a page), pages 0 and 2 resident with their host backup deferred,
    pages 1 and 3 host-only; step 1 fetches rows 4 and 5 (page 1) from host
    into hot slots 0 and 1 (slots 2 and 3 stay empty).  Request 1 is
    admitted from its host copy, 10 rows, every complete page resident."""
    monkeypatch.setattr(oracle, "lib", lambda: poke_lib)
    p = oracle.OraclePool(R, S, T, B, E, PR, MAX_ROWS, CAP)
    rows0 = dhs_workload.payload_rows(TAG, 0, 0, 0, 18, E)
    assert p.admit_device(0, 0, 18, np.array([1, 0, 1, 0], np.uint8), rows0) == (0, 0)
    rows1 = dhs_workload.payload_rows(TAG, 0, 1, 0, 10, E)
    assert p.admit(1, 0, 10, None, rows1) == (0, 0)
    rc, loc, cnt = p.resolve(1, 0, 0, np.array([4, 5, 16], np.int32))
    assert rc == 0 and cnt[5] == 2  # two host fetches
    tags, stamps, page_slot, _ = p.state(0, 0)
    assert list(tags) == [4, 5, -1, -1] and list(stamps) == [1, 1, 0, 0]
    assert list(page_slot[:5]) == [0, -1, 1, -1, -1]
    assert p.check(0, 0) == 0 and p.check(1, 0) == 0
    yield p, poke_lib
    p.close()


def poke(lib, p, r, field, i, v):
    assert lib.orc_test_poke(p._h, r, 0, field, i, v) == 0


def test_valid_states_pass(pool):
    p, lib = pool
    assert p.backup(10) == (0, 2)  # pages 0 and 2 of request 0
    assert p.check(0, 0) == 0 and p.check(1, 0) == 0
    assert p.reclaim([0], 1) == (0, 2)
    assert p.check(0, 0) == 0 and p.check(1, 0) == 0


@pytest.mark.parametrize("field,i,v,want", [
    (TAG_F, 2, 18, 1),     # tag = L: outside [0, L)
    (TAG_F, 2, -2, 1),     # neither a row nor the empty mark
    (STAMP_F, 3, 5, 2),    # empty slot with a stamp
    (STAMP_F, 0, 0, 3),    # row 4 held with stamp 0
    (TAG_F, 1, 4, 4),      # row 4 in slots 0 and 1
])
def test_hot_cache_checks_fire(pool, field, i, v, want):
    p, lib = pool
    poke(lib, p, 0, field, i, v)
    assert p.check(0, 0) == want
    assert p.check(1, 0) == 0


def test_incomplete_page_ready_fires_5(pool):
    p, lib = pool
    # page 4 holds rows 16..19 of an 18-row history: not complete
    poke(lib, p, 0, PAGE_SLOT_F, 4, 2)
    poke(lib, p, 0, SLOT_PAIR_F, 2, 0)
    poke(lib, p, 0, SLOT_PAGE_F, 2, 4)
    assert p.check(0, 0) == 5


@pytest.mark.parametrize("how", ["other_pair", "other_page", "past_capacity"])
def test_foreign_optional_slot_fires_6(pool, how):
    p, lib = pool
    if how == "other_pair":   # slot 0 handed to request 1 in the slot table
        poke(lib, p, 0, SLOT_PAIR_F, 0, 1)
    elif how == "other_page":  # page 1 pointed at page 0's slot
        poke(lib, p, 0, PAGE_SLOT_F, 1, 0)
    else:
        poke(lib, p, 0, PAGE_SLOT_F, 0, CAP)
    assert p.check(0, 0) == 6


def test_page_neither_ready_nor_backed_fires_7(pool):
    """Page 0 dropped from the device while its backup is still deferred:
    its rows are on neither side."""
    p, lib = pool
    poke(lib, p, 0, PAGE_SLOT_F, 0, -1)
    assert p.check(0, 0) == 7


def test_backed_and_pending_fires_8(pool):
    p, lib = pool
    poke(lib, p, 0, BACKED_F, 2, 1)
    assert p.check(0, 0) == 8


def test_backed_without_its_rows_fires_9(pool):
    """Page 2 marked backed up without the copy: the host rows still differ
    from the rows the device holds."""
    p, lib = pool
    poke(lib, p, 0, PEND_F, 2, 0)
    poke(lib, p, 0, BACKED_F, 2, 1)
    assert p.check(0, 0) == 9


def test_host_row_changed_after_backup_fires_9(pool):
    """After the real backup the host copy is right; corrupting one element of
    page 0's host rows breaks the invariant again."""
    p, lib = pool
    assert p.backup(10) == (0, 2)
    assert p.check(0, 0) == 0
    poke(lib, p, 0, HOST_F, 3 * E + 1, 0x1234)
    assert p.check(0, 0) == 9

"""Mutation harness for the CPU oracle: are its pins strong enough?

Each mutant is a copy of oracle/dhs_oracle.c with one plausible mistake
planted (an off-by-one boundary, a wrong tie order, a dropped step, a wrong
ordering rule).  The oracle's pin tests run against every copy in a
subprocess (DHS_ORACLE_SRC points the oracle module at the copy); a mutant is
killed when some pin fails or the mutated oracle crashes.  Every mutant must
be killed, except those listed
as equivalent, which no input can tell apart from the oracle (each says
why).  The pins themselves live in the other test_oracle_*.py files.

Passages the mutants break: "Adaptive DHiSparse", How it works -- Memory
split (complete pages, capacity rule, lowest free slot), Resolution (tail
before the optional map, B-bounded scan, LRU victims, host copy), Speculative
state (one union per verify block; the drafter's ring-buffer window),
Resident-first admission and
Reclamation and refill (backup order, backup before free, bounded
round-robin refill), Limits (decode rows written through to the host).
"""
import concurrent.futures
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PINS = ["test_oracle_pins.py", "test_oracle_bruteforce.py", "test_oracle_union.py",
        "test_oracle_backup.py", "test_oracle_check.py", "test_oracle_loadstep.py"]

# (name, text in dhs_oracle.c, replacement, scope) -- scope: a function whose
# body the replacement is limited to, or None for the whole file
MUTANTS = [
    ("tail_boundary", "if (row >= L - T) return", "if (row > L - T) return", None),
    ("range_lets_L_through", "if (row < 0 || row >= L) return ORC_NO_LOC;",
     "if (row < 0 || row > L) return ORC_NO_LOC;", None),
    ("ring_index", "(uint32_t)(pair * T + row % T)", "(uint32_t)(pair * T + (row + 1) % T)",
     None),
    ("lru_tie_highest_slot", "if (best < 0 || st[j] < st[best]) best = j;",
     "if (best < 0 || st[j] <= st[best]) best = j;", None),
    ("budget_off_by_one", "  if (n_miss > avail) {", "  if (n_miss > avail + 1) {", None),
    ("hit_not_stamped", "      st[j] = step;\n      c_hot++;", "      c_hot++;", None),
    ("stamps_not_committed", "  memcpy(src->stamps, st, sizeof(uint32_t) * (size_t)B);",
     "  (void)0;", None),
    ("evicted_counts_empty", "    if (src->tags[best] != -1) evicted++;", "    evicted++;",
     None),
    ("scan_count_off_by_one",
     "      if ((uint32_t)(j + 1) > scan_max) scan_max = (uint32_t)(j + 1);",
     "      if ((uint32_t)j > scan_max) scan_max = (uint32_t)j;", None),
    ("erange_drops_step1",
     "      for (int64_t f = 0; f < n; ++f) loc[f] = step1_location(p, src, pair, sel[f]);",
     "      for (int64_t f = 0; f < n; ++f) loc[f] = ORC_NO_LOC;", None),
    ("ebudget_drops_step1",
     "    for (int64_t e = 0; e < n; ++e) loc[e] = step1_location(p, src, pair, sel[e]);",
     "    for (int64_t e = 0; e < n; ++e) loc[e] = ORC_NO_LOC;", None),
    ("no_host_write_through",
     "      if (!src->window) memcpy(src->host + (size_t)row * E, rows + (size_t)j * E, E * 2);",
     "      (void)0;", None),
    ("allocator_highest_slot", "for (int64_t i = p->first_free; i < p->capacity; ++i)",
     "for (int64_t i = p->capacity - 1; i >= 0; --i)", None),
    ("reclaim_order_reversed", "  for (int32_t i = 0; i < n && got < deficit; ++i) {",
     "  for (int32_t i = n - 1; i >= 0 && got < deficit; --i) {", None),
    ("capacity_ignores_reserve", "  if (p->used + want > p->capacity - p->reserve) {",
     "  if (p->used + want > p->capacity) {", None),
    ("no_backup_before_free", "        if (!src->backed[q]) backup_page(src, p, q);",
     "        (void)0;", None),
    ("backup_newest_first", "src->pend[q] < best->pend[best_q]",
     "src->pend[q] > best->pend[best_q]", None),
    ("refill_cursor_stuck", "  p->rr = r;", "  (void)r;", None),
    ("refill_ignores_reserve",
     "while (n < max_pages && p->used < p->capacity - p->reserve && idle < p->R)",
     "while (n < max_pages && p->used < p->capacity && idle < p->R)", None),
    ("device_admission_marks_backed", "    src->backed[q] = 0;\n    src->pend[q] = ++p->bseq;",
     "    src->pend[q] = 0;", None),
    ("optional_rows_from_host_copy",
     "      from = (o->imported ? o->imported : o->host) + (size_t)row * E;",
     "      from = o->host + (size_t)row * E;", None),
    ("union_per_query_layout", "      loc[u] = per_entry[e];", "      loc[e] = per_entry[e];",
     None),
    ("window_lower_bound_off_by_one",
     "const int64_t lo = src->window && L > p->T ? L - p->T : 0;",
     "const int64_t lo = src->window && L > p->T ? L - p->T - 1 : 0;", None),
    ("window_admission_ring_slot", "      int64_t row = N - m + j;",
     "      int64_t row = N - m + j + 1;", None),
    ("window_serves_whole_history",
     "const int64_t lo = src->window && L > p->T ? L - p->T : 0;",
     "const int64_t lo = 0;", None),
] + [
    # each invariant check of orc_check taken out in turn
    (f"check_{k}_removed", f"return {k};", ";", "int orc_check(") for k in range(1, 10)
]

# Mutants no input can distinguish from the oracle.
EQUIVALENT = [
    # Step 1 tests that an optional page is complete before using the map;
    # admission and refill only ever give complete pages a slot, so a ready
    # map entry always belongs to a complete page and the test is redundant.
    ("page_completeness_in_step1",
     "if ((page + 1) * PR <= N && src->page_slot[page] >= 0)",
     "if (page * PR < N && src->page_slot[page] >= 0)", None),
]


def plant(text, old, new, scope):
    start = text.index(scope) if scope else 0
    head, tail = text[:start], text[start:]
    assert tail.count(old) >= 1, f"mutation site not found: {old!r}"
    if scope is None:
        assert text.count(old) == 1, f"mutation site not unique: {old!r}"
    return head + tail.replace(old, new, 1)


def run_pins(src_path):
    env = dict(os.environ, DHS_ORACLE_SRC=src_path)
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
           "-m", "not gpu"] + [os.path.join(HERE, f) for f in PINS]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    failed = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED")]
    return r.returncode, failed[:1]


def test_every_mutant_is_killed(tmp_path, oracle_lib, gen_lib):
    with open(oracle.source_path()) as f:
        original = f.read()
    jobs = {}
    for name, old, new, scope in MUTANTS + EQUIVALENT:
        d = tmp_path / name
        d.mkdir()
        path = d / "dhs_oracle.c"
        path.write_text(plant(original, old, new, scope))
        jobs[name] = str(path)
    workers = max(1, min(8, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        res = dict(zip(jobs, ex.map(run_pins, jobs.values())))
    survivors = [n for n, _, _, _ in MUTANTS if res[n][0] == 0]
    assert not survivors, f"mutants not killed by any pin: {survivors}"
    for n, _, _, _ in MUTANTS:
        # a failed pin (exit 1) or a crash of the mutated oracle (a signal:
        # e.g. an eviction with no victim left writes out of bounds)
        assert res[n][0] == 1 or res[n][0] < 0, f"{n}: pytest exit {res[n][0]}"
    for n, _, _, _ in EQUIVALENT:
        assert res[n][0] == 0, f"{n} is listed as equivalent but a pin kills it: {res[n][1]}"

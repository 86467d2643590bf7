"""Benchmark of the hierarchical sparse KV resolve + gather decode step.

One step = append every source's decode rows, resolve every request's
selections through tail / optional map / hot cache / pinned host, and
gather every layer into staging, over one batch of a synthetic workload
(default: the C64 speculative-verify workload -- 64 requests x 4 layers x
32K-row histories of 576 bf16, 8 verify queries of top-k 2048 each, B 4096,
40 % of complete pages optional-resident, misses fetched from pinned host
memory; the largest per-step work of the single-GPU workloads).

The bench cycles through the workload's decode steps; after the last one
the pool is reset (every request released and admitted again, untimed) and
the sequence starts over, so any number of genuine decode steps can be
timed.  A workload's own warm-up steps (C128: 16) and the first step after
every reset (hot caches empty) always run untimed.

Prints one JSON line.  value = selected rows resolved + gathered per second
with every input resident in HBM: device time from CUDA events on the
launching stream.  L2: a workload whose step moves less than four times the
L2 size (C8, Tiny) is timed with L2 flushed before every step (a 256 MB
write, then a 256 MB read of another buffer); the others have inputs far
larger than L2 and are timed as consecutive steps (--l2 overrides).  The
line carries the other method's figure too.  A second pass times the same
steps through dhs_resolve and dhs_gather separately, so the gather kernel's
own duration gives the roofline.  e2e = the same metric through the C ABI
with each step's selections and decode rows copied from pinned host memory
and its locations + counters read back, copies inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c64]
  python bench.py --impl reference ...   (the CPU oracle as the reference arm)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("selected KV rows resolved+gathered/sec and GB/s vs HBM & host-link "
          "roofline")
UNIT = "rows/s"
L2_BYTES = 129 << 20  # GB300 L2, about 129 MB
GATHER_WRITE_BYTES_PER_ENTRY = 1152 + 4  # staging row write + location read
# host-buffer pipeline depth: output sets a serving loop cycles through (the
# host reads step s-3's outputs after enqueuing step s).  C8, µs a step with
# 2 / 3 / 4 / 6 sets: 31.0 / 28.4 / 27.9 / 27.9
E2E_SETS = 4


_ALG_CACHE = {}


def gather_alg_bytes(cfg, wl, step, union=False):
    key = (cfg, step, union)
    if key not in _ALG_CACHE:
        _ALG_CACHE[key] = _gather_alg_bytes(cfg, wl, step, union)
    return _ALG_CACHE[key]


def _gather_alg_bytes(cfg, wl, step, union=False):
    """Algorithmic HBM bytes of one step's gather launch: every unique
    selected row of a resolved (request, source) read once (verify queries
    and reuse layers read the same rows again), and every gathered entry
    written to staging with its location read.  Union staging writes each
    layer's distinct rows once and still reads every entry's location."""
    import numpy as np
    sel = wl.selections()[step - 1]  # [R][sel_sources][Q][k]
    flat = np.sort(sel.reshape(sel.shape[0], sel.shape[1], -1), axis=-1)
    # distinct rows of each (request, selection source)
    u = 1 + np.count_nonzero(np.diff(flat, axis=-1), axis=-1)
    if u.shape[1] != cfg.sources:  # one selection shared by every source
        u = np.repeat(u, cfg.sources, axis=1)
    reads = int(u.sum())
    writes = int(u.sum() + cfg.reuse_layers * u[:, 0].sum()) if union else 0
    if not union:
        return reads * cfg.row_bytes + cfg.entries_per_step * GATHER_WRITE_BYTES_PER_ENTRY
    return (reads + writes) * cfg.row_bytes + cfg.entries_per_step * 4


def l2_flushed(args, cfg, wl) -> bool:
    """Whether timed steps start from a flushed L2: --l2, or (auto) when the
    gather's algorithmic bytes per step, averaged over the cycle, are below
    four times the L2 size -- otherwise every step's inputs are far larger
    than L2 and steps are timed back to back.  Both arms take the same
    decision, so their configurations match."""
    if args.l2 != "auto":
        return args.l2 == "flush"
    probe = Cycle(cfg, None)
    steps = [s for s in range(1, cfg.total_steps + 1) if probe.timed(s)]
    mean = sum(gather_alg_bytes(cfg, wl, s, args.union) for s in steps) / len(steps)
    return mean < 4 * L2_BYTES


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 3000 on c8/tiny, 320 otherwise)")
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--config", default="c64")
    ap.add_argument("--l2", default="auto", choices=["auto", "flush", "none"],
                    help="L2 between timed steps: flushed, or consecutive steps; auto = "
                         "flush when a step moves less than 4x the L2 size")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--copy-ctas", type=int, default=0)
    ap.add_argument("--resolve-paired", type=int, default=-1,
                    help="DHS_OPT_RESOLVE_PAIRED: -1 auto, 0 one 1024-thread CTA per SM, 1 "
                         "512-thread CTAs two per SM whenever they fit")
    ap.add_argument("--copy-pdl", type=int, default=-1,
                    help="DHS_OPT_COPY_PDL: -1 auto, 0 copy after the resolve grid, 1 overlapped")
    ap.add_argument("--copy-steal", type=int, default=-1,
                    help="DHS_OPT_COPY_STEAL: -1 auto, 0 each copy block keeps to its own items, "
                         "1 rows claimed through per-item cursors")
    ap.add_argument("--gather-impl", type=int, default=1)
    ap.add_argument("--stage-misses", type=int, default=1,
                    help="DHS_OPT_STAGE_MISSES: 1 = the host copy writes fetched rows into staging")
    ap.add_argument("--early", type=int, default=1,
                    help="DHS_OPT_EARLY: 1 = fused gathers copy rows before the grids end")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=5.0)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--kernel-steps", type=int, default=500)
    ap.add_argument("--trace-steps", type=int, default=100)
    ap.add_argument("--b2b-steps", type=int, default=200,
                    help="steps timed with the other L2 method (step_hbm), 0 = none")
    ap.add_argument("--no-hugepages", action="store_true")
    ap.add_argument("--gemm", type=int, default=4096,
                    help="--experiment prefetch: per-layer compute, an n x n x n bf16 GEMM")
    ap.add_argument("--union", action="store_true",
                    help="union verification staging (DHS_ITEM_UNION)")
    ap.add_argument("--experiment", default=None, choices=["loadstep", "prefetch"],
                    help="run an experiment instead of the benchmark (one JSON line)")
    return ap.parse_args()


def workload_desc(cfg, union=False, flushed=True):
    return {
        "staging": ("union: each distinct row of a verify block staged once, plus "
                    "per-query index lists") if union else "per query [Q][k] rows",
        "workload": (f"{cfg.name}: {cfg.requests} requests x {cfg.layers} layers "
                     f"({cfg.sources} KV sources), {cfg.history}-row histories of "
                     f"{cfg.row_elems} bf16, top-k {cfg.topk} x {cfg.queries} queries, "
                     f"B {cfg.hot}, tail {cfg.tail}, {cfg.total_steps}-step cycle"),
        "requests": cfg.requests, "sources": cfg.sources, "layers": cfg.layers,
        "history_rows": cfg.history, "topk": cfg.topk, "queries": cfg.queries,
        "hot_rows": cfg.hot, "tail_rows": cfg.tail,
        "residency": cfg.residency if cfg.residency is not None else
        f"admission-driven, pool {cfg.capacity_frac:.0%} of pages",
        "entries_per_step": cfg.entries_per_step,
        "l2": ("flushed before every timed step (256 MB write, then a read of another 256 MB)"
               if flushed else
               "not flushed: consecutive steps, each moving far more than the L2 size "
               "(inputs larger than L2)"),
        "cold_steps": "the first step after each pool reset runs untimed (hot caches empty)",
    }


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, device) -> float:
    """Max of a per-rank float over all ranks (identity without a process
    group).  The timed duration of a step sequence is the slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class Cycle:
    """Next decode step of a workload, resetting after its last step.  A
    workload's own warm-up steps, and at least the first step after a reset
    (every hot cache empty, which a serving pool meets only for newly
    admitted requests), are not timed."""

    def __init__(self, cfg, reset, cold=1):
        self.cfg, self.reset, self.s = cfg, reset, 0
        self.untimed = max(cfg.warmup_steps, min(cold, cfg.total_steps - 1))

    def next(self):
        if self.s == self.cfg.total_steps:
            self.reset()
            self.s = 0
        self.s += 1
        return self.s

    def timed(self, s):
        return s > self.untimed


# ---------------------------------------------------------------- CPU oracle

class OracleTimer:
    """The CPU oracle as it stands, one thread per group of requests (ctypes
    releases the GIL inside the oracle); threads run each step together and
    wall time is taken around the step."""

    # host memory the oracle's own copies of the sampled requests' rows may take
    SAMPLE_BYTES = 8 << 30

    def __init__(self, cfg, wl, threads=None, union=False):
        from oracle.run import OracleRun
        self.cfg = cfg
        per_request = cfg.sources * cfg.max_rows * cfg.row_bytes
        cores = os.cpu_count() or 1
        # a bounded sample: requests are independent once admitted, so the
        # oracle simulates the first n (all of them when they fit)
        n = max(1, min(cfg.requests, max(cores, 8), self.SAMPLE_BYTES // per_request))
        reqs = list(range(n))
        self.sampled = n
        self.threads = threads or min(n, cores)
        self.runs = [OracleRun(cfg, wl, requests=reqs[i::self.threads], union=union)
                     for i in range(self.threads)]
        self.cycle = Cycle(cfg, self._reset)

    @property
    def rows_per_step(self):
        """Selected rows the sampled requests resolve + gather per step."""
        return self.cfg.entries_per_step * self.sampled // self.cfg.requests

    def _reset(self):
        for r in self.runs:
            r.reset()

    def step(self):
        """Run untimed warm-up steps as needed, then one timed step; returns
        its wall seconds."""
        s = self.cycle.next()
        while not self.cycle.timed(s):
            self._run(s)
            s = self.cycle.next()
        t0 = time.perf_counter()
        self._run(s)
        return time.perf_counter() - t0

    def _run(self, s):
        ts = [threading.Thread(target=r.step, args=(s,)) for r in self.runs]
        for t in ts:
            t.start()
        for t in ts:
            t.join()

    def close(self):
        for r in self.runs:
            r.pool.close()


def run_reference(args, cfg):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    from dhs_workload.configs import Workload
    wl = Workload(cfg)
    flushed = l2_flushed(args, cfg, wl)
    ot = OracleTimer(cfg, wl, union=args.union)
    for _ in range(args.warmup):
        ot.step()
    K = args.steps
    dt = sum(ot.step() for _ in range(K))
    ot.close()
    value = K * ot.rows_per_step / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": K, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": workload_desc(cfg, args.union, flushed),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": ot.threads,
                         "kind": "oracle",
                         "sample": f"{K} decode steps of the workload, requests 0-{ot.sampled - 1} "
                                   f"of {cfg.requests}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)  # first sample lands before the timed region
        except OSError:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.perf_counter(), ln.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, power, reasons = [], None, [], set()
        for t, ln in self.lines:
            if not (t0 <= t <= t1 + 0.06):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(self.NAMES, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": statistics.median(power) if power else None}


# ---------------------------------------------------------------- our arm

def traffic_from_profile(kernel_src: str, profile: str):
    """Per-launch DRAM bytes of the gather kernel from a committed ncu summary,
    valid only while the kernel source is unchanged since the capture."""
    try:
        with open(profile) as f:
            data = json.load(f)
        with open(kernel_src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()[:16]
        if data.get("kernel_sha256_16") != digest:
            return None
        return data.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        return None


def h2d_peak_gbs(dev, nbytes=1 << 30, reps=5):
    """Pinned host -> device copy bandwidth (cudaMemcpyAsync via torch), best
    of `reps`: the host-link roofline for the copy kernel."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize(dev)
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    return best


def traced_pass(run, cycle, steps, dev, flush_l2, trace, alone=False):
    """Kernel timeline of `steps` fused steps (DHS_OPT_TRACE into `trace`,
    int64[8] allocated beforehand; synchronised per step -- not the
    headline): per-kernel durations, and the host-copy kernel's bytes and
    time for the host-link roofline (aggregate, and the median step's).
    alone: each step's append + resolve + host copy only, no gather (the
    copy without the gather's traffic beside it)."""
    import torch
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    cfg = run.cfg
    run.pool.set_option(dhs.DHS_OPT_TRACE, trace.data_ptr())
    res, cp, ga, lt, span, host_b, copy_s = [], [], [], [], [], 0, 0.0
    rates = []
    for _ in range(steps):
        s = cycle.next()
        while not cycle.timed(s):
            run.step(s)
            s = cycle.next()
        flush_l2()
        trace[0::2] = (1 << 63) - 1
        trace[1::2] = 0
        if alone:
            run.append(s)
            run.resolve(s)
        else:
            run.step(s)
        torch.cuda.synchronize(dev)
        t = trace.cpu().tolist()
        hb = int(run.counters[..., 5].sum().item()) * cfg.row_bytes
        res.append((t[1] - t[0]) / 1e3)
        if t[5] > t[4] > 0:
            ga.append((t[5] - t[4]) / 1e3)
        end = max(t[1], t[3], t[5])
        if t[7] > t[6] > 0:  # fresh-row list copy
            lt.append((t[7] - t[6]) / 1e3)
            end = max(end, t[7])
        span.append((end - t[0]) / 1e3)
        if t[3] > t[2] > 0:
            cp.append((t[3] - t[2]) / 1e3)
            if hb:
                host_b += hb
                copy_s += (t[3] - t[2]) / 1e9
                rates.append(hb / (t[3] - t[2]))
    run.pool.set_option(dhs.DHS_OPT_TRACE, 0)
    med = statistics.median
    return {"resolve_us": med(res), "gather_us": med(ga) if ga else None,
            "copy_us": med(cp) if cp else None,
            "copy_us_max": max(cp) if cp else None,
            "fresh_list_us": med(lt) if lt else None,
            "step_span_us": med(span),
            "host_bytes_per_step": host_b / steps,
            "copy_gbs": (host_b / copy_s / 1e9) if copy_s else None,
            "copy_gbs_median_step": med(rates) if rates else None}


def measure_e2e(run, cycle, steps, dev, stream):
    """The metric through the C ABI with host buffers for `steps` further
    decode steps.  Each step copies its selections and decode rows in from
    pinned host memory (one block), runs, and copies its locations +
    counters (+ union indices) back to pinned host memory (one block), all
    inside the timed region.

    value: pipelined as a serving loop runs it.  dhs_decode_step_host_async
    puts each step's input copy on an input stream and its output copy on an
    output stream, so inputs come in and earlier steps' outputs go out while
    a step runs.  Device output blocks and host output buffers cycle through
    E2E_SETS sets; after enqueuing step s the host waits for step
    s - (E2E_SETS - 1)'s outputs (an event) and reads its counters, so the
    host's own work per step overlaps the device's instead of following it.
    A set is rewritten only after the host has read its previous outputs, and
    every step has its own device input block, so no device-side waits are
    needed.  Wall clock over runs of consecutive steps (a workload's pool
    reset between cycles is outside it), all of a run's outputs read inside
    it.
    sync_value: one blocking dhs_decode_step_host call per step, wall clock
    around each call."""
    import numpy as np
    import torch
    T = run.cfg.total_steps
    in_host = [run.step_in[s].cpu().pin_memory() for s in range(T)]
    D = E2E_SETS
    blocks = [run.output_block(i) for i in range(D)]

    def span(dst, src):
        return (dst.data_ptr(), src.data_ptr(), src.numel() * src.element_size())

    cnt_off = run.counters.data_ptr() - run.step_out.data_ptr()
    sets = []  # host outputs of each device output block
    for blk in blocks:
        out_h = torch.empty(blk.shape, dtype=torch.uint8).pin_memory()
        cnt_h = out_h[cnt_off:cnt_off + run.counters.numel() * 4].view(torch.int32)
        sets.append((cnt_h.view(run.counters.shape).numpy(), [span(out_h, blk)], out_h))
    # the calls' arguments for every step of the cycle, built once as a caller would
    io = [[run.host_io(s, [span(run.step_in[s - 1], in_host[s - 1])], sets[b][1], out_set=b)
           for s in range(1, T + 1)] for b in range(D)]

    def next_timed():
        s = cycle.next()
        while not cycle.timed(s):
            run.step(s)
            s = cycle.next()
        return s

    # the allocations above changed the page tables: untimed steps re-warm
    # the host copy's translations before anything is timed
    for _ in range(3):
        run.step(next_timed())
    # blocking calls
    torch.cuda.synchronize(dev)
    sync_dt = 0.0
    for _ in range(steps):
        s = next_timed()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        run.step_host(s, io=io[0][s - 1])
        sync_dt += time.perf_counter() - t0
    # pipelined: runs of consecutive steps up to the end of the cycle
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    out_done = [torch.cuda.Event() for _ in range(D)]  # each set's output copy
    dt, n, seen = 0.0, 0, 0
    while n < steps:
        seg = [next_timed()]
        while len(seg) < steps - n and seg[-1] < T:
            seg.append(next_timed())
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for j, s in enumerate(seg):
            b = j % D  # its last outputs (step j - D) were read at iteration j - 1
            run.step_host(s, io=io[b][s - 1], wait=False, in_stream=s_in, out_stream=s_out)
            out_done[b].record(s_out)
            if j >= D - 1:  # step j - (D - 1)'s outputs are in host memory: read them
                k = (j - (D - 1)) % D
                out_done[k].synchronize()
                seen += int(sets[k][0][..., 0].sum(dtype=np.int64))
        for j in range(max(0, len(seg) - (D - 1)), len(seg)):
            out_done[j % D].synchronize()
            seen += int(sets[j % D][0][..., 0].sum(dtype=np.int64))
        dt += time.perf_counter() - t0
        n += len(seg)
    torch.cuda.synchronize(dev)
    c = run.cfg
    want = steps * c.requests * c.sources * c.queries * c.topk
    if seen != want:  # counters[0] = entries each resolved (request, source) took
        raise RuntimeError(f"e2e outputs: {seen} entries counted, {want} expected")
    return {"value": c.entries_per_step * steps / dt, "unit": UNIT,
            "h2d_bytes_per_step": int(in_host[0].numel()),
            "d2h_bytes_per_step": int(run.step_out.numel()),
            "steps": steps, "seconds": dt,
            "sync_value": c.entries_per_step * steps / sync_dt,
            "path": f"dhs_decode_step_host_async per step: input copy on an input stream, "
                    f"step, output copy on an output stream ({D} output sets); after "
                    f"enqueuing step s, step s-{D - 1}'s outputs waited for and read; "
                    "sync_value: blocking dhs_decode_step_host, one call per step"}


def run_loadstep(args):
    """The load-step on/off experiment through the C ABI: host-fetched
    fraction of unique selected rows per phase with optional residency on
    and off, decode-step device time per phase, and the admission
    machinery's copy rates (device admission, deferred backup, refill)."""
    import torch
    from dhs_workload.loadstep import LOADSTEP, phase_fractions, run
    from hierarchical_sparse_kv_dhs_gb300.runner import LoadStepGpu
    cfg = LOADSTEP
    out = {"experiment": "loadstep", "data": "synthetic",
           "config": {"slots": cfg.slots, "low_load_requests": cfg.low,
                      "sources": cfg.sources, "history_rows": cfg.history,
                      "topk": cfg.topk, "hot_rows": cfg.hot, "tail_rows": cfg.tail,
                      "optional_pages": cfg.capacity,
                      "steps": [cfg.steps_low, cfg.steps_burst, cfg.steps_drain],
                      "refill_pages_per_step": cfg.refill_per_step,
                      "backup_pages_per_step": cfg.backup_per_step}}
    for mode in ("on", "off"):
        g = LoadStepGpu(cfg.topk)
        recs = run(g, cfg, residency=(mode == "on"))
        fr = phase_fractions(recs)
        step_us = {}
        for ph in ("low", "burst", "drain"):
            ts = [t for t, x in zip(g.times["step"], recs) if x["phase"] == ph]
            step_us[ph] = statistics.median(ts) * 1e6 if ts else None
        rates = {k: (g.bytes[k] / sum(g.times[k]) / 1e9) if g.times[k] else None
                 for k in ("admit", "backup", "refill")}
        out[mode] = {"host_fraction": fr, "step_us_median": step_us,
                     "copy_gbs": rates,
                     "pages_moved": {k: g.bytes[k] // (cfg.page_rows * cfg.row_elems * 2)
                                     for k in ("backup", "refill")},
                     "resident_pages_end_of_phase": {
                         ph: [x for x in recs if x["phase"] == ph][-1]["resident_pages"]
                         for ph in ("low", "burst", "drain")}}
        g.close()
        del g
        torch.cuda.empty_cache()
    print(json.dumps(out), flush=True)


def set_pool_options(run, args):
    """The pool options that the command line sets (library defaults otherwise)."""
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    if args.copy_ctas:
        run.pool.set_option(dhs.DHS_OPT_COPY_CTAS, args.copy_ctas)
    run.pool.set_option(dhs.DHS_OPT_COPY_PDL, args.copy_pdl)
    if args.copy_steal != -1:
        run.pool.set_option(dhs.DHS_OPT_COPY_STEAL, args.copy_steal)
    run.pool.set_option(dhs.DHS_OPT_RESOLVE_PAIRED, args.resolve_paired)
    run.pool.set_option(dhs.DHS_OPT_GATHER_IMPL, args.gather_impl)
    run.pool.set_option(dhs.DHS_OPT_EARLY, args.early)
    run.pool.set_option(dhs.DHS_OPT_STAGE_MISSES, args.stage_misses)


def run_prefetch(args, cfg):
    """Per-layer decode with the caller's compute between layers (a bf16
    GEMM standing in for each layer's attention + MLP), two schedules over
    the same steps from the same pool state:
      serial    per layer: resolve, gather, compute (pool stream);
      prefetch  layer 0 resolved on the pool stream, every later resolving
                layer by dhs_prefetch on a side stream at step start; per
                layer: gather, compute;
      pipelined as prefetch, with every gather on a second stream
                (dhs_gather_on), overlapping the previous layer's compute.
    Device time per step from CUDA events on the pool stream."""
    import torch
    from dhs_workload.configs import Workload
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun
    wl = Workload(cfg)
    run = GpuRun(cfg, wl)
    set_pool_options(run, args)
    n = args.gemm
    A = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
    B = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
    C = torch.empty(n, n, device="cuda", dtype=torch.bfloat16)
    layers = list(range(len(run.layers)))
    resolving = [l for l, (kind, _) in enumerate(run.layers) if kind == "resolve"]

    def serial(step):
        run.append(step)
        for l in layers:
            if l in resolving:
                run.resolve_layer(step, l)
            run.gather_layer(step, l)
            torch.mm(A, B, out=C)

    def prefetch(step):
        run.append(step)
        run.resolve_layer(step, layers[0])
        if len(resolving) > 1:
            run.prefetch_layers(step, resolving[1:])
        for l in layers:
            run.gather_layer(step, l)
            torch.mm(A, B, out=C)

    gs = torch.cuda.Stream()
    main = torch.cuda.current_stream()

    def pipelined(step):
        # prefetch, and every layer's gather on a second stream so that it
        # overlaps the previous layer's compute
        run.append(step)
        run.resolve_layer(step, layers[0])
        if len(resolving) > 1:
            run.prefetch_layers(step, resolving[1:])
        for l in layers:
            run.gather_layer(step, l, stream=gs)
            ev = torch.cuda.Event()
            ev.record(gs)
            main.wait_event(ev)
            torch.mm(A, B, out=C)

    def compute_only():
        for _ in layers:
            torch.mm(A, B, out=C)

    out = {"experiment": "prefetch", "config": workload_desc(cfg), "gemm": [n, n, n],
           "layers": len(layers), "resolving_layers": len(resolving)}
    for name, fn in (("serial", serial), ("prefetch", prefetch), ("pipelined", pipelined),
                     ("compute_only", None)):
        run.reset()
        torch.cuda.synchronize()
        ts = []
        for step in range(1, cfg.total_steps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            if fn is None:
                compute_only()
            else:
                fn(step)
            e1.record()
            e1.synchronize()
            if step > cfg.warmup_steps + 2:
                ts.append(e0.elapsed_time(e1) * 1e3)
        rc, flags = run.status()
        if rc != 0:
            raise RuntimeError(f"device status {rc} flags {flags}")
        out[name + "_us_median"] = statistics.median(ts)
    out["hidden_us"] = out["serial_us_median"] - out["prefetch_us_median"]
    out["hidden_pipelined_us"] = out["serial_us_median"] - out["pipelined_us_median"]
    run.close()
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.experiment == "loadstep":
        run_loadstep(args)
        return
    if args.experiment == "prefetch":
        from dhs_workload.configs import CONFIGS
        run_prefetch(args, CONFIGS[args.config])
        return
    from dhs_workload.configs import CONFIGS
    cfg = CONFIGS[args.config]
    if args.steps is None:
        args.steps = 3000 if cfg.name in ("c8", "tiny") else 320
    if args.impl == "reference":
        run_reference(args, cfg)
        return
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K, W = args.steps, args.warmup

    from dhs_workload.configs import Workload
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun

    wl = Workload(cfg)
    run = GpuRun(cfg, wl, device=dev, hugepages=not args.no_hugepages, union=args.union)
    set_pool_options(run, args)
    stream = torch.cuda.current_stream(dev)
    # Every device buffer the bench uses is allocated here, before any step
    # is timed: a new device allocation changes the GPU's page tables, and
    # the host copy after it re-walks the translations of the pinned host
    # region (a cold copy, like the first one after admission).
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clean64 = torch.zeros(32 << 20, dtype=torch.int64, device=dev)  # 256 MB
    trace = torch.zeros(8, dtype=torch.int64, device=dev)
    ctx_src = torch.empty(cfg.entries_per_step * cfg.row_bytes, dtype=torch.uint8, device=dev)
    ctx_dst = torch.empty_like(ctx_src)
    tiny = torch.zeros(1, dtype=torch.int32, device=dev)
    h2d = h2d_peak_gbs(dev)

    def flush_l2():
        # write 256 MB (evicts the previous step's lines and writes back its
        # dirty ones), then read another 256 MB so that L2 holds only clean
        # lines whose eviction costs the timed step nothing
        flush.zero_()
        clean64.sum()

    # One calibration cycle from the admitted state (every cycle after a
    # reset repeats it exactly): the host fetches of each step, for the
    # step's algorithmic bytes.  It also warms the kernels up.
    T = cfg.total_steps
    host_rows_of = {}
    for s in range(1, T + 1):
        run.step(s)
        torch.cuda.synchronize(dev)
        host_rows_of[s] = int(run.counters[..., 5].sum().item())
    rc, flags = run.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} flags {flags} during calibration")
    run.reset()
    cycle = Cycle(cfg, run.reset)
    timed_of = [s for s in range(1, T + 1) if cycle.timed(s)]
    gather_alg = {s: gather_alg_bytes(cfg, wl, s, args.union) for s in timed_of}
    # the whole step: the gather's bytes, every resolved entry's selection
    # read, and each host fetch's write into its hot slot
    step_alg = {s: gather_alg[s] + cfg.resolved_per_step * 4 + host_rows_of[s] * cfg.row_bytes
                for s in timed_of}
    flushed = l2_flushed(args, cfg, wl)

    def next_timed():
        s = cycle.next()
        while not cycle.timed(s):
            run.step(s)
            s = cycle.next()
        return s

    def time_steps(n, with_flush):
        """Device ms of each of n further timed steps and the steps run.
        with_flush: L2 flushed before every step, events around each step;
        else runs of consecutive steps (to the end of the cycle), an event
        after each step."""
        ms, steps = [], []
        while len(steps) < n:
            if with_flush:
                s = next_timed()
                flush_l2()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run.step(s)  # dhs_decode_step: append + resolve + gather
                e1.record(stream)
                ms.append((e0, e1))
                steps.append(s)
                continue
            seg = [next_timed()]
            while len(seg) < n - len(steps) and seg[-1] < T:
                seg.append(next_timed())
            torch.cuda.synchronize(dev)
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(seg) + 1)]
            evs[0].record(stream)
            for j, s in enumerate(seg):
                run.step(s)
                evs[j + 1].record(stream)
            torch.cuda.synchronize(dev)
            ms += list(zip(evs[:-1], evs[1:]))
            steps += seg
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in ms], steps

    for _ in range(W):
        run.step(next_timed())
    rc, flags = run.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} flags {flags} during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    step_ms, steps_run = time_steps(K, flushed)
    t_wall1 = time.perf_counter()
    if world > 1:
        torch.distributed.barrier()
    clock_info = clocks.stop(t_wall0, t_wall1)
    rc, flags = run.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} flags {flags} in the timed region")
    total_s = reduce_max(sum(step_ms) / 1e3, dev)
    entries = cfg.entries_per_step
    value = world * entries * K / total_s

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "of measured" if peak else "of fallback"
    peak = peak or 6800.0

    def step_level(ms, steps):
        """The whole step's algorithmic HBM bytes over its device time."""
        gbs = sum(step_alg[s] for s in steps) / (sum(ms) / 1e3) / 1e9
        srt = sorted(ms)
        # position in the workload's cycle: the early steps after each pool
        # reset fill the hot caches again (and the host copy's translations)
        early = [m for m, s in zip(ms, steps) if s <= T // 2]
        late = [m for m, s in zip(ms, steps) if s > T // 2]
        halves = {"us_median_first_half_of_cycle":
                  statistics.median(early) * 1e3 if early else None,
                  "us_median_second_half_of_cycle":
                  statistics.median(late) * 1e3 if late else None}
        return {**halves, "us_per_step_mean": sum(ms) * 1e3 / len(ms),
                "us_per_step_median": statistics.median(ms) * 1e3,
                "us_per_step_p90": srt[min(len(srt) - 1, int(0.9 * len(srt)))] * 1e3,
                "us_per_step_max": srt[-1] * 1e3,
                "rows_per_s": entries * len(ms) / (sum(ms) / 1e3),
                "alg_GBps": gbs, "hbm_frac": gbs / peak, "steps": len(ms)}

    # The other L2 method, for comparison (breakdown)
    other_ms, other_steps = (time_steps(min(K, args.b2b_steps), not flushed)
                             if args.b2b_steps else (None, None))
    step_hbm = {("flushed" if flushed else "back_to_back"): step_level(step_ms, steps_run)}
    if other_ms:
        step_hbm["back_to_back" if flushed else "flushed"] = step_level(other_ms, other_steps)
    step_hbm["bytes"] = ("per step: the gather's algorithmic bytes (each distinct selected "
                         "row read once, every entry's staging row written and location "
                         "read), every resolved entry's 4-byte selection read, and 1152 B "
                         "per host fetch written into its hot slot")
    step_hbm["peak"] = f"{peak} GB/s hbm_gbs {peak_src}"
    maybe_flush = flush_l2 if flushed else (lambda: None)

    # Kernel timing pass (not the headline): the same steps through
    # dhs_resolve then dhs_gather, events around each, so the gather kernel
    # (the byte-dominant one) is timed alone for the roofline.
    K2 = min(K, args.kernel_steps)
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K2)]
    k_steps = []
    for i in range(K2):
        s = next_timed()
        k_steps.append(s)
        maybe_flush()
        ev2[i][0].record(stream)
        run.append(s)
        run.resolve(s)
        ev2[i][1].record(stream)
        run.gather(s)
        ev2[i][2].record(stream)
    torch.cuda.synchronize(dev)
    gather_ms = [e[1].elapsed_time(e[2]) for e in ev2]
    resolve_ms = [e[0].elapsed_time(e[1]) for e in ev2]

    # Context for the gather's roofline, timed the same way (flush, events):
    # a contiguous device copy of the staging bytes, and one trivial launch
    ctx_n = min(K2, 100)
    src_b, dst_b = ctx_src, ctx_dst
    ctx = {}
    for name, fn in (("contiguous_copy_us", lambda: dst_b.copy_(src_b)),
                     ("empty_launch_us", lambda: tiny.fill_(0))):
        evc = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(ctx_n)]
        for i in range(ctx_n):
            flush_l2()
            evc[i][0].record(stream)
            fn()
            evc[i][1].record(stream)
        torch.cuda.synchronize(dev)
        ctx[name] = statistics.median(e[0].elapsed_time(e[1]) * 1e3 for e in evc)
    ctx["contiguous_copy_GBps"] = 2 * src_b.numel() / (ctx["contiguous_copy_us"] * 1e3)
    ctx["what"] = (f"cudaMemcpyAsync device-to-device of {src_b.numel()} contiguous bytes "
                   "(the step's staging bytes) and a 1-element fill, medians of "
                   f"{ctx_n}, L2 flushed before each")
    # two untimed steps re-warm whatever the copy context left cold
    for _ in range(2):
        run.step(next_timed())
    trace_info = traced_pass(run, cycle, min(K, args.trace_steps), dev, maybe_flush, trace)
    alone_info = traced_pass(run, cycle, min(K, args.trace_steps), dev, maybe_flush, trace,
                             alone=True)
    link = None
    if trace_info["copy_gbs"]:
        link = {"bound": "host link (NVLink-C2C)", "kernel": "hostcopy",
                "achieved": trace_info["copy_gbs"], "peak": h2d, "unit": "GB/s",
                "frac": trace_info["copy_gbs"] / h2d,
                "peak_source": "measured in this run: pinned H2D cudaMemcpyAsync, 1 GiB",
                "bytes_per_step": trace_info["host_bytes_per_step"],
                "copy_us": trace_info["copy_us"],
                "achieved_median_step": trace_info["copy_gbs_median_step"],
                "alone": {"achieved": alone_info["copy_gbs"],
                          "frac": (alone_info["copy_gbs"] or 0.0) / h2d,
                          "copy_us": alone_info["copy_us"],
                          "what": "the same steps' append + resolve + host copy without the "
                                  "gather running beside the copy"},
                "timed": (f"{min(K, args.trace_steps)} traced fused steps "
                          f"({'L2 flushed before each' if flushed else 'no flush'}): "
                          "host bytes fetched / span of the copy kernel's copying "
                          "(%globaltimer)")}

    cnt = run.counters.cpu().numpy().reshape(-1, 8).astype("int64")
    tiers = {"unique": int(cnt[:, 1].sum()), "tail": int(cnt[:, 2].sum()),
             "optional": int(cnt[:, 3].sum()), "hot": int(cnt[:, 4].sum()),
             "host": int(cnt[:, 5].sum())}
    host_rows = tiers["host"]

    e2e = None
    if args.e2e_steps:
        e2e = measure_e2e(run, cycle, args.e2e_steps, dev, stream)
        e2e["value"] = world * entries * args.e2e_steps / reduce_max(e2e["seconds"], dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ot = OracleTimer(cfg, wl, union=args.union)
        dt, n = 0.0, 0
        while dt < args.cpu_seconds:
            dt += ot.step()
            n += 1
        ot.close()
        cpu = {"value": n * ot.rows_per_step / dt, "unit": UNIT, "cores": ot.threads,
               "kind": "oracle",
               "sample": f"{n} decode steps of the same workload, requests 0-{ot.sampled - 1} "
                         f"of {cfg.requests} ({n * ot.rows_per_step} rows, {dt:.1f} s timed), "
                         f"{ot.threads} threads"}
        # the same oracle on one thread, a shorter sample
        ot1 = OracleTimer(cfg, wl, threads=1, union=args.union)
        dt1, n1 = 0.0, 0
        while dt1 < args.cpu_seconds / 2:
            dt1 += ot1.step()
            n1 += 1
        ot1.close()
        cpu["single_thread_value"] = n1 * ot1.rows_per_step / dt1
        cpu["single_thread_sample"] = f"{n1} decode steps, {dt1:.1f} s timed, 1 thread"

    gather_avg = sum(gather_ms) / K2 / 1e3
    alg_bytes = sum(gather_alg[s] for s in k_steps) / K2  # per launch, averaged
    achieved = alg_bytes / gather_avg / 1e9
    gather_src = "gather.cu"
    traffic = traffic_from_profile(
        os.path.join(ROOT, "hierarchical_sparse_kv_dhs_gb300", "csrc", gather_src),
        os.path.join(ROOT, "profiles", f"gather_{cfg.name}_traffic.json"))
    n_resolve = -(-cfg.requests * cfg.sources // 256)
    n_gather = -(-cfg.requests * cfg.layers // 384)
    # the fresh-row list copy launches only for gather-only (Reuse) items the
    # host copy does not write itself: beyond three per resolved item
    fresh = int(run.pool.get_option(dhs.DHS_OPT_FRESH_LIST) and cfg.reuse_layers > 3)
    # append folded into resolve; resolve + host copy per chunk, the gathers,
    # and the fresh-row list copy when it is on
    launches = K * (2 * n_resolve + n_gather + fresh)
    impl = ["vector", "tma"][args.gather_impl]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": sum(step_ms) / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8", "data": "synthetic",
        "config": workload_desc(cfg, args.union, flushed),
        "roofline": {"bound": "hbm", "kernel": f"gather_{impl}", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"hbm_gbs {peak_src} (copy, read+write bytes)",
                     "traffic": traffic, "alg_bytes_per_launch": alg_bytes,
                     "traffic_note": "DRAM bytes inside one launch (ncu): every row is read "
                                     "from DRAM, but staging rows still in L2 when the "
                                     "launch ends are written back after it, by the next "
                                     "step's traffic or the flush",
                     "timed": f"{K2} launches, CUDA events around dhs_gather "
                              + ("(L2 flushed before each step)" if flushed else
                                 "(consecutive steps, no flush)"),
                     "context": ctx},
        "host_link": link,
        "step_hbm": step_hbm,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clock_info,
        "breakdown": {
            "path": f"dhs_decode_step (append folded into resolve; resolve, host copy "
                    f"and gather PDL-overlapped{', fresh-row list copy' if fresh else ''}), "
                    f"gather {impl}",
            "step_ms_median": statistics.median(step_ms),
            "traced_kernel_us": trace_info,
            "h2d_peak_gbs": h2d,
            "split_append_resolve_hostcopy_ms": sum(resolve_ms) / K2,
            "split_gather_ms": sum(gather_ms) / K2,
            "wall_s_timed_region": t_wall1 - t_wall0,
            "last_step_unique_rows": tiers,
            "last_step_host_bytes": host_rows * cfg.row_bytes,
        },
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    run.close()
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

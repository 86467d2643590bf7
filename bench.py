"""Benchmark of the hierarchical sparse KV resolve + gather decode step.

One step = append every source's decode rows + resolve every request's
selections through tail / optional map / hot cache / pinned host + gather
every layer into staging, over one batch of a synthetic workload (default:
the C8 decode workload, 8 requests x 4 layers x 32K-row histories, top-k
2048, B 4096, all imported history optional-resident).

Prints one JSON line.  value = selected rows resolved + gathered per second
with every input resident in HBM, device time from CUDA events on the
launching stream, L2 flushed (a 256 MB write) before every timed step.
e2e = the same metric through the C ABI with the step's selections and
decode rows copied from pinned host buffers and the locations + counters
read back, host<->device copies inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c8]
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
GATHER_BYTES_PER_ENTRY = 1152 + 1152 + 4  # row read + row write + location read


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--config", default="c8")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--copy-ctas", type=int, default=0)
    ap.add_argument("--gather-impl", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-sample-steps", type=int, default=None)
    ap.add_argument("--e2e-steps", type=int, default=16)
    return ap.parse_args()


def workload_desc(cfg):
    return {
        "workload": (f"{cfg.name}: {cfg.requests} requests x {cfg.layers} layers "
                     f"({cfg.sources} KV sources), {cfg.history}-row histories of "
                     f"{cfg.row_elems} bf16, top-k {cfg.topk} x {cfg.queries} queries, "
                     f"B {cfg.hot}, tail {cfg.tail}"),
        "requests": cfg.requests, "sources": cfg.sources, "layers": cfg.layers,
        "history_rows": cfg.history, "topk": cfg.topk, "queries": cfg.queries,
        "hot_rows": cfg.hot, "tail_rows": cfg.tail,
        "residency": cfg.residency if cfg.residency is not None else
        f"admission-driven, pool {cfg.capacity_frac:.0%} of pages",
        "entries_per_step": cfg.entries_per_step,
        "l2": "flushed (256 MB write) before every timed step",
    }


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------- reference arm

def oracle_sample(cfg, wl, steps, requests=None, threads=None):
    """Time the CPU oracle (as it stands) on `steps` steps of the workload,
    one thread per request (ctypes releases the GIL inside the oracle).
    Returns (rows/s, threads, entries, seconds)."""
    from oracle.run import OracleRun
    requests = list(range(cfg.requests)) if requests is None else requests
    threads = threads or min(len(requests), os.cpu_count() or 1)
    runs = []
    groups = [requests[i::threads] for i in range(threads)]
    for g in groups:
        runs.append(OracleRun(cfg, wl, requests=g))

    def work(run):
        for step in range(1, steps + 1):
            run.step(step)

    t0 = time.perf_counter()
    ts = [threading.Thread(target=work, args=(r,)) for r in runs]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    dt = time.perf_counter() - t0
    for r in runs:
        r.pool.close()
    entries = len(requests) * cfg.layers * cfg.queries * cfg.topk * steps
    return entries / dt, threads, entries, dt


def run_reference(args, cfg):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    from dhs_workload.configs import Workload
    wl = Workload(cfg)
    steps = args.steps or 2
    sample_steps = min(cfg.total_steps, max(1, steps))
    value, threads, entries, dt = oracle_sample(cfg, wl, sample_steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": sample_steps, "warmup": 0,
        "ms_per_step": dt * 1e3 / sample_steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": workload_desc(cfg),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"all {cfg.requests} requests, steps 1..{sample_steps}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


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


def main():
    args = parse()
    from dhs_workload.configs import CONFIGS
    base = CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, base)
        return
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    K = args.steps if args.steps is not None else max(1, base.steps - args.warmup)
    W = args.warmup
    E = 0 if args.no_e2e else args.e2e_steps
    # decode steps of the run: the workload's own warm-up, then W untimed,
    # K timed and E end-to-end steps of the same workload shape
    cfg = base.scaled(steps=W + K + E)
    from dhs_workload.configs import Workload
    from hierarchical_sparse_kv_dhs_gb300 import dhs
    from hierarchical_sparse_kv_dhs_gb300.runner import GpuRun

    wl = Workload(cfg)
    run = GpuRun(cfg, wl, device=dev)
    if args.copy_ctas:
        run.pool.set_option(dhs.DHS_OPT_COPY_CTAS, args.copy_ctas)
    if args.gather_impl:
        run.pool.set_option(dhs.DHS_OPT_GATHER_IMPL, args.gather_impl)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    first = cfg.warmup_steps  # the workload's own warm-up steps run untimed
    for s in range(1, first + W + 1):
        run.step(s)
    rc, flags = run.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} flags {flags} during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t_wall0 = time.perf_counter()
    for i in range(K):
        s = first + W + 1 + i
        flush.zero_()
        ev[i][0].record(stream)
        run.append(s)
        run.resolve(s)
        ev[i][1].record(stream)
        run.gather(s)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    clock_info = clocks.stop()
    rc, flags = run.status()
    if rc != 0:
        raise RuntimeError(f"device status {rc} flags {flags} in the timed region")
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    gather_ms = [e[1].elapsed_time(e[2]) for e in ev]
    resolve_ms = [e[0].elapsed_time(e[1]) for e in ev]
    total_s = sum(step_ms) / 1e3
    if world > 1:
        t = torch.tensor([total_s], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_s = float(t.item())
    entries = cfg.entries_per_step
    value = world * entries * K / total_s

    # counters of the last step: where rows resolved
    cnt = run.counters.cpu().numpy().reshape(-1, 8).astype("int64")
    tiers = {"unique": int(cnt[:, 1].sum()), "tail": int(cnt[:, 2].sum()),
             "optional": int(cnt[:, 3].sum()), "hot": int(cnt[:, 4].sum()),
             "host": int(cnt[:, 5].sum())}
    host_bytes = tiers["host"] * cfg.row_bytes

    # ---------------- e2e through the C ABI with host buffers
    e2e = None
    if E:
        e2e = measure_e2e(run, cfg, first + W + K + 1, E, dev, stream)
        if world > 1:
            t = torch.tensor([e2e["seconds"]], dtype=torch.float64, device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            e2e["value"] = world * cfg.entries_per_step * E / float(t.item())

    # ---------------- CPU baseline (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample_steps = args.cpu_sample_steps or min(8, cfg.total_steps)
        v, threads, n_entries, dt = oracle_sample(cfg, wl, sample_steps)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"all {cfg.requests} requests x {cfg.layers} layers, steps "
                         f"1..{sample_steps} ({n_entries} rows, {dt:.1f} s)"}

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    gather_avg = sum(gather_ms) / K / 1e3
    alg_bytes = entries * GATHER_BYTES_PER_ENTRY
    achieved = alg_bytes / gather_avg / 1e9
    traffic = traffic_from_profile(
        os.path.join(ROOT, "hierarchical_sparse_kv_dhs_gb300", "csrc", "gather.cu"),
        os.path.join(ROOT, "profiles", f"gather_{cfg.name}_traffic.json"))
    n_resolve_launches = -(-cfg.requests * cfg.sources // 256)
    n_gather_launches = -(-cfg.requests * cfg.layers // 512)
    launches = K * (1 + 2 * n_resolve_launches + n_gather_launches)
    step_bytes = alg_bytes + cfg.resolved_per_step * 4  # + selections read
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": sum(step_ms) / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8", "data": "synthetic", "config": workload_desc(cfg),
        "roofline": {"bound": "hbm", "kernel": "gather", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} (hbm_gbs, copy read+write)",
                     "traffic": traffic,
                     "alg_bytes_per_launch": alg_bytes},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clock_info,
        "breakdown": {
            "append_resolve_hostcopy_ms": sum(resolve_ms) / K,
            "gather_ms": sum(gather_ms) / K,
            "step_GBps_alg": step_bytes / (sum(step_ms) / K / 1e3) / 1e9,
            "wall_s_timed_region": t_wall,
            "last_step_unique_rows": tiers,
            "last_step_host_bytes": host_bytes,
        },
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    run.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_e2e(run, cfg, first, steps, dev, stream):
    """Same metric through the C ABI for `steps` further decode steps: each
    step's selections and decode rows are copied from pinned host memory,
    the step runs, and its locations + counters are read back into pinned
    host memory (wall clock, synchronised per step as a caller reading its
    result would be)."""
    import torch
    last = first + steps - 1
    sel_host = [run.sel[s - 1].cpu().pin_memory() for s in range(first, last + 1)]
    rows_host = [run.app_rows[s - 1].cpu().pin_memory() for s in range(first, last + 1)]
    loc_host = torch.empty(run.loc.shape, dtype=run.loc.dtype).pin_memory()
    cnt_host = torch.empty(run.counters.shape, dtype=run.counters.dtype).pin_memory()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i, s in enumerate(range(first, last + 1)):
        run.sel[s - 1].copy_(sel_host[i], non_blocking=True)
        run.app_rows[s - 1].copy_(rows_host[i], non_blocking=True)
        run.step(s)
        loc_host.copy_(run.loc, non_blocking=True)
        cnt_host.copy_(run.counters, non_blocking=True)
        stream.synchronize()
    dt = time.perf_counter() - t0
    h2d = sel_host[0].numel() * 4 + rows_host[0].numel() * 2
    d2h = loc_host.numel() * 4 + cnt_host.numel() * 4
    return {"value": cfg.entries_per_step * steps / dt, "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "seconds": dt}


if __name__ == "__main__":
    main()

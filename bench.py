"""Benchmark: store + load of a hybrid KDA + MLA cache between a paged GPU
pool and per-chunk objects, through liblmc's C ABI.

One step = the whole hot path over one batch: the store (gather every whole
chunk of every request into per-object-group objects) and the load (scatter
every object into a fresh pool under new block tables). The default workload
is Kimi-Linear's 24-layer hybrid (18 KDA + 6 MLA, N = 944, padded layout,
chunk = N) with 32 requests of 8192 tokens: 11.67 GB of objects per
direction. Metric: bytes moved per second, each payload byte read once and
written once (2 x payload per store, 2 x payload per load).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1] [--impl reference]

Under torchrun each rank runs its own copy of the workload on its own GPU
(independent requests, no exchange between ranks); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "store/load GB/s moved and % of GB300 HBM peak; chunks/sec per config"
NOMINAL_HBM_GBS = 7900.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def _kernel_sha():
    h = hashlib.sha256()
    with open(os.path.join(ROOT, "state_cache_paging_gb300", "csrc", "paging.cu"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str, workload_index: int):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    entry = t.get(f"config{workload_index}", {}).get(kernel)
    if not entry or entry.get("kernel_sha") != _kernel_sha():
        return None
    return entry.get("dram_bytes_per_launch")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait(timeout=10)

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        self.out.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.out.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _dist():
    if int(os.environ.get("WORLD_SIZE", "1")) <= 1:
        return None, 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    world = int(os.environ["WORLD_SIZE"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    return dist, rank, world, local


# ----------------------------------------------------------------------------
# CPU oracle leg (cpu_baseline and --impl reference)
# ----------------------------------------------------------------------------

def oracle_sample(cfg_index: int, requests: int, reps: int, threads: int, warmup: int = 1):
    """Times the CPU oracle's store + load on a bounded sample of the workload
    (the first `requests` requests), `threads` workers over disjoint jobs."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    cfg = W.CONFIGS[cfg_index]
    C = oracle.negotiate_chunk(cfg.requested_chunk, cfg.N)
    ids = list(range(min(requests, cfg.num_requests)))
    inp = W.make_inputs(cfg, functools.partial(oracle.layout, cfg.layers, cfg.N, cfg.packed), C, ids)
    L = inp.layout
    import torch
    pool = W.fill_normal(torch.empty(L.pool_bytes, dtype=torch.uint8), cfg.seed).numpy()
    fresh = np.full(L.pool_bytes, W.SENTINEL, dtype=np.uint8)
    arena = np.zeros(inp.arena_bytes, dtype=np.uint8)
    # split every group's jobs into `threads` disjoint slices
    parts = [[J[k::threads] for J in inp.jobs] for k in range(threads)]
    payload = inp.payload_bytes
    with ThreadPoolExecutor(threads) as ex:
        for _ in range(warmup):
            list(ex.map(lambda p: oracle.store(L, C, pool, inp.tables_src, p, arena), parts))
            list(ex.map(lambda p: oracle.load(L, C, fresh, inp.tables_dst, p, arena), parts))
        t0 = time.perf_counter()
        for _ in range(reps):
            assert all(s == 0 for s in ex.map(lambda p: oracle.store(L, C, pool, inp.tables_src, p, arena), parts))
            assert all(s == 0 for s in ex.map(lambda p: oracle.load(L, C, fresh, inp.tables_dst, p, arena), parts))
        dt = time.perf_counter() - t0
    chunks = sum(int(x) // C for x in inp.lengths)
    gbs = 4 * payload * reps / dt / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"first {len(ids)} of {cfg.num_requests} requests ({payload} payload bytes per direction), "
                      f"{reps} timed store+load passes after {warmup} warm-up, {threads} threads over disjoint jobs",
            "chunks_per_s": round(chunks * reps / dt, 2), "seconds": round(dt, 3)}


def run_reference(args):
    dist, rank, world, local = _dist()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    cfg = W.CONFIGS[args.config]
    # each step is one store + load pass over a bounded sample (8 of the 32
    # requests); warm-up passes run inside the same call before timing starts
    res = oracle_sample(args.config, requests=8, reps=args.steps, threads=threads, warmup=args.warmup)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["seconds"] * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": cfg.name, "index": cfg.index, "sample": res["sample"]},
        "cpu_baseline": {k: res[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": res["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "chunks_per_s": res["chunks_per_s"]}))


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def run_gpu(args):
    import torch

    import state_cache_paging_gb300 as lmc

    dist, rank, world, local = _dist()
    if dist is not None:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = W.CONFIGS[args.config]
    if cfg.mixed:
        raise SystemExit("the mixed step is measured by --config 4 in bench_mixed mode only")

    C = lmc.lmc_negotiate_chunk(cfg.requested_chunk, cfg.N)
    ids = list(range(cfg.num_requests)) if args.requests is None else list(range(args.requests))
    # each rank runs its own independent copy of the batch (weak scaling)
    build = functools.partial(lmc.lmc_layout_build, cfg.layers, cfg.N, cfg.packed)
    inp = W.make_inputs(cfg, build, C, ids)
    L = inp.layout
    payload = inp.payload_bytes
    chunks = sum(int(x) // C for x in inp.lengths)

    pool = torch.empty(L.pool_bytes, dtype=torch.uint8, device=dev)
    W.fill_normal(pool, cfg.seed + 101 * rank)
    fresh = torch.full((L.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=dev)
    arena = torch.empty(inp.arena_bytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t_src = [torch.from_numpy(t).to(dev) for t in inp.tables_src]
    t_dst = [torch.from_numpy(t).to(dev) for t in inp.tables_dst]
    jobs = [lmc.jobs_to_device(j, dev) for j in inp.jobs]
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        lmc.lmc_store(L, C, pool, t_src, jobs, arena, status, stream)
        if ev is not None:
            ev[1].record(stream)
        lmc.lmc_load(L, C, fresh, t_dst, jobs, arena, status, stream)
        if ev is not None:
            ev[2].record(stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step()
    barrier()
    assert int(status.item()) == 0, f"device status {int(status.item()):#x}"

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        t_start.record(stream)
        for k in range(args.steps):
            step(evs[k])
        t_end.record(stream)
        barrier()
    clocks = clk.summary()
    total_ms = t_start.elapsed_time(t_end)
    store_ms = [e[0].elapsed_time(e[1]) for e in evs]
    load_ms = [e[1].elapsed_time(e[2]) for e in evs]
    assert int(status.item()) == 0

    # end to end through the public API with host buffers: per step, the
    # block tables and jobs go host -> device, the stored objects go device ->
    # host (the host cache tier), come back host -> device and are loaded.
    host_arena = torch.empty(inp.arena_bytes, dtype=torch.uint8, pin_memory=True)
    host_tables = [torch.from_numpy(t).pin_memory() for t in inp.tables_src + inp.tables_dst]
    host_jobs = [torch.from_numpy(np.ascontiguousarray(j).view(np.uint8)).pin_memory() for j in inp.jobs]
    host_status = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    dev_tables = t_src + t_dst
    h2d = sum(t.numel() * 4 for t in host_tables) + sum(j.numel() for j in host_jobs) + inp.arena_bytes
    d2h = inp.arena_bytes + 4

    def e2e_step():
        for h, d in zip(host_tables, dev_tables):
            d.copy_(h, non_blocking=True)
        for h, d in zip(host_jobs, jobs):
            d.copy_(h, non_blocking=True)
        lmc.lmc_store(L, C, pool, t_src, jobs, arena, status, stream)
        host_arena.copy_(arena, non_blocking=True)
        arena.copy_(host_arena, non_blocking=True)
        lmc.lmc_load(L, C, fresh, t_dst, jobs, arena, status, stream)
        host_status.copy_(status, non_blocking=True)

    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(2):
        e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    assert int(host_status.item()) == 0
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    ms_per_step = total_ms / args.steps
    if dist is not None:
        t = torch.tensor([ms_per_step, e2e_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_per_step, e2e_ms = float(t[0]), float(t[1])
    if rank != 0:
        dist.destroy_process_group()
        return

    bytes_per_step = 4 * payload  # store and load each read and write every payload byte
    value = bytes_per_step * world / (ms_per_step * 1e-3) / 1e9
    peak, peak_src = _peaks()
    st_avg, ld_avg = statistics.mean(store_ms), statistics.mean(load_ms)
    dominant, dom_ms = ("store", st_avg) if st_avg >= ld_avg else ("load", ld_avg)
    achieved = 2 * payload / (dom_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": cfg.name, "index": cfg.index, "requests": len(ids),
                   "payload_bytes_per_direction": payload, "chunk": C, "N": cfg.N,
                   "layout": "packed" if cfg.packed else "padded", "pool_bytes": L.pool_bytes,
                   "l2": "inputs larger than L2 (pool and objects are each > 11 GB; no flush)",
                   "parallelism": f"{world} independent replica(s), no exchange"},
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "pct_of_nominal_hbm": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "chunks_per_s": round(chunks * world / (ms_per_step * 1e-3), 1),
        "store": {"ms": round(st_avg, 4), "gbs": round(2 * payload / (st_avg * 1e-3) / 1e9, 2)},
        "load": {"ms": round(ld_avg, 4), "gbs": round(2 * payload / (ld_avg * 1e-3) / 1e9, 2)},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 2), "peak": peak,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs: copy read+write)",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": _traffic(dominant, cfg.index),
                     "algorithmic_bytes_per_launch": 2 * payload},
        "e2e": {"value": round(bytes_per_step * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        line["cpu_baseline"] = oracle_sample(args.config, requests=8, reps=20, threads=threads)
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--requests", type=int, default=None, help="use only the first R requests")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--impl", choices=["lmc", "reference"], default="lmc")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

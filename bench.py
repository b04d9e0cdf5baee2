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

The line's headline is that workload. The default run then times the other
workloads (configs 2-4) and operations (the INT8 codec, block-granular
objects, in-pool copies) one after another in the same process, each as its
own entry with CUDA-event times, clocks and roofline (`--no-extra-lines`
times the selected one alone). The headline also carries the end-to-end
step (objects through page-locked host memory and back) and the CPU oracle
timed on the same payload.

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


def _traffic(kernel: str, workload_index: int, op: str):
    """The committed small-case ncu capture of `kernel` (its function name)
    on a workload and operation: {"case", "ratio" = DRAM bytes / algorithmic
    bytes, ...}, or None when none was taken or the kernel source changed
    since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    key = f"config{workload_index}" + ("" if op == "paging" else f"/{op}")
    entry = t.get(key, {}).get(kernel)
    if not entry or entry.get("kernel_sha") != _kernel_sha() or not entry.get("ratio"):
        return None
    return entry


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


def _kernel_times(nbytes, ms_list):
    """Mean (the line's figure), median and best of one kernel's per-step
    CUDA-event times, with the bytes-moved rates they give."""
    if not ms_list or max(ms_list) <= 0:
        return {"ms": None, "gbs": None, "bytes": nbytes}
    mean, med, best = statistics.mean(ms_list), statistics.median(ms_list), min(ms_list)
    return {"ms": round(mean, 4), "gbs": _gbs(nbytes, mean), "bytes": nbytes, "median_ms": round(med, 4),
            "median_gbs": _gbs(nbytes, med), "best_ms": round(best, 4), "best_gbs": _gbs(nbytes, best)}


def _with_frac(times, peak):
    """A kernel's mean rate as a fraction of the HBM peak (each kernel of a
    line, beside the roofline of the slower one)."""
    times["frac_of_peak"] = round(times["gbs"] / peak, 4) if times.get("gbs") else None
    return times


def _gbs(nbytes, ms):
    return round(nbytes / (ms * 1e-3) / 1e9, 2) if nbytes and ms > 0 else None


def _all_ranks(dist, flag: bool, device) -> bool:
    """True when `flag` holds on every rank (a MIN over ranks; the local
    flag when there is no process group)."""
    if dist is None:
        return bool(flag)
    import torch
    t = torch.tensor([1 if flag else 0], dtype=torch.int32, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return bool(t.item())


def _reduce_max(dist, values, device):
    """Max over ranks of per-rank timings (the only cross-rank step)."""
    import torch
    t = torch.tensor(values, device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


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

def _host_free_bytes() -> int:
    """Free host memory (sysconf), the budget for the oracle's buffers."""
    return os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")


def _step_requests(cfg, requests=None) -> int:
    """Requests one step moves: all of the workload, or one wave when the
    workload runs in waves (config 3: one 131,072-token request per wave),
    or the first `requests`."""
    if requests is not None:
        return min(requests, cfg.num_requests)
    return cfg.num_requests // cfg.waves if cfg.waves > 1 else cfg.num_requests


def _workload_config(cfg, op, n_req, store_payload, load_payload, C, pool_bytes, world):
    """The `config` object of a line; the GPU arm and the oracle arm print
    the same one for the same workload."""
    scope = (f"one wave: {n_req} of {cfg.num_requests} requests ({cfg.waves} waves of the workload)"
             if cfg.waves > 1 and n_req * cfg.waves == cfg.num_requests else
             f"{n_req} of {cfg.num_requests} requests")
    return {"workload": cfg.name, "index": cfg.index, "op": op, "requests": n_req, "scope": scope,
            "store_payload_bytes": int(store_payload), "load_payload_bytes": int(load_payload),
            "chunk": int(C), "N": cfg.N, "layout": "packed" if cfg.packed else "padded",
            "pool_bytes": int(pool_bytes),
            "l2": "inputs larger than L2 (pool and objects are each many GB; no flush)",
            "parallelism": f"{world} independent replica(s), no exchange"}


def _oracle_footprint(inp) -> int:
    L = inp.layout
    if inp.cfg.mixed:
        return L.pool_bytes + inp.load_arena_bytes + inp.store_arena_bytes
    return 2 * L.pool_bytes + inp.arena_bytes


def oracle_time(cfg_index: int, n_req: int, threads: int, seconds: float = 10.0, reps: int | None = None,
                warmup: int = 1, pool_of=None):
    """Times the CPU oracle, as written, on the first `n_req` requests of a
    workload (the payload of one GPU step): the store of every whole chunk
    then the load into a fresh pool under new tables (the mixed step: its
    load of cached chunks and its store of new chunks on one pool), with
    `threads` workers over disjoint jobs. `reps` timed passes after `warmup`
    (or as many as fill about `seconds`). Host memory is checked first
    (sysconf); when the buffers do not fit, the requests run in consecutive
    waves and the times add up. Pool bytes: pool_of(inputs) when given (the
    GPU arm's own device pool), else seeded N(0,1) draws on the host."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    cfg = W.CONFIGS[cfg_index]
    C = oracle.negotiate_chunk(cfg.requested_chunk, cfg.N)
    build = functools.partial(oracle.layout, cfg.layers, cfg.N, cfg.packed)
    ids = list(range(n_req))
    budget = int(0.6 * _host_free_bytes())
    full = W.make_inputs(cfg, build, C, ids)
    n_waves = 1
    while n_waves < len(ids) and max(
            _oracle_footprint(W.make_inputs(cfg, build, C, list(w)))
            for w in np.array_split(np.array(ids), n_waves)) > budget:
        n_waves += 1
    waves = [list(map(int, w)) for w in np.array_split(np.array(ids), n_waves) if len(w)]
    total_s, passes, payload, chunks, store_total, load_total = 0.0, None, 0, 0, 0, 0
    for w in waves:
        inp = full if len(waves) == 1 else W.make_inputs(cfg, build, C, w)
        L = inp.layout
        pool = pool_of(inp) if (pool_of is not None and len(waves) == 1) else \
            W.fill_normal_host(L.pool_bytes, cfg.seed, threads)
        sizes = inp.object_bytes
        if cfg.mixed:
            src = W.fill_normal_host(inp.load_arena_bytes, cfg.seed + 7, threads)
            out = np.zeros(inp.store_arena_bytes, dtype=np.uint8)
            lparts = [[J[k::threads] for J in inp.load_jobs] for k in range(threads)]
            sparts = [[J[k::threads] for J in inp.store_jobs] for k in range(threads)]
            loaded = sum(int(sizes[g]) * len(j) for g, j in enumerate(inp.load_jobs))
            stored = sum(int(sizes[g]) * len(j) for g, j in enumerate(inp.store_jobs))

            def one_pass(ex):
                a = list(ex.map(lambda p: oracle.load(L, C, pool, inp.tables_src, p, src), lparts))
                b = list(ex.map(lambda p: oracle.store(L, C, pool, inp.tables_src, p, out), sparts))
                return a + b
            units = sum(len(j) for j in inp.store_jobs) // max(1, L.num_object_groups)
        else:
            fresh = np.full(L.pool_bytes, W.SENTINEL, dtype=np.uint8)
            arena = np.zeros(inp.arena_bytes, dtype=np.uint8)
            parts = [[J[k::threads] for J in inp.jobs] for k in range(threads)]
            loaded = stored = inp.payload_bytes

            def one_pass(ex):
                a = list(ex.map(lambda p: oracle.store(L, C, pool, inp.tables_src, p, arena), parts))
                b = list(ex.map(lambda p: oracle.load(L, C, fresh, inp.tables_dst, p, arena), parts))
                return a + b
            units = sum(int(x) // C for x in inp.lengths)
        with ThreadPoolExecutor(threads) as ex:
            t0 = time.perf_counter()
            for _ in range(max(1, warmup)):
                assert all(st == 0 for st in one_pass(ex))
            per_pass = (time.perf_counter() - t0) / max(1, warmup)
            if passes is None:
                passes = reps if reps is not None else int(min(100, max(2, seconds / len(waves) / per_pass)))
            t0 = time.perf_counter()
            for _ in range(passes):
                assert all(st == 0 for st in one_pass(ex))
            total_s += time.perf_counter() - t0
        payload += loaded + stored
        store_total += stored
        load_total += loaded
        chunks += units
        del pool
    gbs = 2 * payload * passes / total_s / 1e9  # each payload byte read once and written once
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"the whole step: {n_req} of {cfg.num_requests} requests, {payload} object bytes moved per "
                      f"pass (store + load) in {len(waves)} wave(s) of host buffers, {passes} timed passes after "
                      f"{max(1, warmup)} warm-up, {threads} thread(s) over disjoint jobs",
            "chunks_per_s": round(chunks * passes / total_s, 2), "seconds": round(total_s, 3),
            "passes": passes, "waves": len(waves), "payload_bytes_per_pass": payload,
            "config": _workload_config(cfg, "paging", n_req, store_total, load_total, C, full.layout.pool_bytes, 1)}


def run_reference(args):
    dist, rank, world, local = _dist()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    cfg = W.CONFIGS[args.config]
    n_req = _step_requests(cfg, args.requests)
    # each step is one store + load pass over the GPU step's whole payload;
    # the warm-up passes run inside the same call before timing starts
    res = oracle_time(args.config, n_req, threads, reps=args.steps, warmup=args.warmup)
    config = dict(res["config"], parallelism=f"{world} independent replica(s), no exchange")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["seconds"] * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": config,
        "cpu_baseline": {k: res[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": res["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "chunks_per_s": res["chunks_per_s"]}))


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def split_parts(jobs, object_bytes, parts):
    """Splits packed jobs (ordered by request, chunk, group) into `parts`
    ranges of (request, chunk) units: [(per-group (row0, row1), arena lo, hi)]."""
    units = sorted({(int(j["request"]), int(j["chunk"])) for J in jobs for j in J})
    index = {u: k for k, u in enumerate(units)}
    uid = [np.array([index[(int(j["request"]), int(j["chunk"]))] for j in J], dtype=np.int64) for J in jobs]
    n = len(units)
    bounds = [round(k * n / parts) for k in range(parts + 1)]
    out = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if a == b:
            continue
        rows, lo, hi = [], None, None
        for g, J in enumerate(jobs):
            sel = np.flatnonzero((uid[g] >= a) & (uid[g] < b))
            r0, r1 = (int(sel[0]), int(sel[-1]) + 1) if sel.size else (0, 0)
            rows.append((r0, r1))
            if sel.size:
                lo = int(J["offset"][r0]) if lo is None else min(lo, int(J["offset"][r0]))
                end = int(J["offset"][r1 - 1]) + int(object_bytes[g])
                hi = end if hi is None else max(hi, end)
        if lo is not None:
            out.append((rows, lo, hi))
    return out


def _huge_bytes(m) -> int:
    """Bytes of the mapping `m` backed by transparent huge pages (smaps)."""
    import ctypes
    start = ctypes.addressof(ctypes.c_char.from_buffer(m))
    total, inside = 0, False
    try:
        with open("/proc/self/smaps") as f:
            for line in f:
                head = line.split()[0]
                if "-" in head and ":" not in head:
                    lo, hi = (int(x, 16) for x in head.split("-"))
                    inside = lo <= start < hi
                elif inside and line.startswith("AnonHugePages:"):
                    total += int(line.split()[1]) * 1024
    except OSError:
        return -1
    return total


class HostArena:
    """Page-locked host memory for the objects of the end-to-end step (the
    host cache tier). A single multi-GB cudaHostAlloc buffer can stream
    device -> host at a quarter of the link's rate once earlier processes have
    churned host memory (measured on these boxes: 48 against 193 GB/s), while
    the same bytes in transparent huge pages keep the full rate. So the
    buffer is anonymous memory advised to huge pages, faulted in, and
    registered with CUDA; where that is unavailable, plain pinned memory."""

    def __init__(self, torch, nbytes: int):
        import mmap
        self.torch, self.nbytes, self._map, self._ptr = torch, int(nbytes), None, None
        self.kind = "pinned (cudaHostAlloc)"
        if self.nbytes > 0.85 * _host_free_bytes():
            # faulting the pages in must not run the host out of memory
            raise MemoryError(f"{self.nbytes} bytes of host memory requested, "
                              f"{_host_free_bytes()} free")
        try:
            m = mmap.mmap(-1, max(self.nbytes, 1), flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            m.madvise(mmap.MADV_HUGEPAGE)
            a = np.frombuffer(m, dtype=np.uint8, count=self.nbytes)
            a[::1 << 12] = 0  # fault every page in under the huge-page advice
            try:
                m.madvise(getattr(mmap, "MADV_COLLAPSE", 25))  # gather what stayed in small pages
            except OSError:
                pass
            rc = torch.cuda.cudart().cudaHostRegister(a.ctypes.data, max(self.nbytes, 1), 0)
            if int(getattr(rc, "value", rc)) != 0:
                raise RuntimeError(f"cudaHostRegister: {rc}")
            self._map, self._ptr = m, a.ctypes.data
            self.tensor = torch.from_numpy(a)
            self.kind = f"huge pages ({_huge_bytes(m) / 2**30:.1f} of {self.nbytes / 2**30:.1f} GiB), registered"
        except (AttributeError, OSError, RuntimeError, ValueError):
            self.tensor = torch.empty(self.nbytes, dtype=torch.uint8, pin_memory=True)

    def close(self):
        """Unregisters the memory (after every copy into or out of it is done)."""
        if self._ptr is not None:
            self.torch.cuda.synchronize()
            self.torch.cuda.cudart().cudaHostUnregister(self._ptr)
            self._ptr = None
        self.tensor = None


class PagingStep:
    """Device inputs and one step of the hot path for a workload.

    Plain workloads: the store (pool -> objects) then the load (objects ->
    a fresh pool under new block tables), on one stream. The mixed step
    (one pool): the load of cached chunks and the store of new chunks,
    issued concurrently on two streams that touch disjoint blocks."""

    def __init__(self, lmc, torch, cfg, dev, rank, ids, op="paging"):
        self.lmc, self.torch, self.cfg, self.dev, self.op = lmc, torch, cfg, dev, op
        C = lmc.lmc_negotiate_chunk(cfg.requested_chunk, cfg.N)
        build = functools.partial(lmc.lmc_layout_build, cfg.layers, cfg.N, cfg.packed)
        inp = W.make_inputs(cfg, build, C, ids)
        if op == "q8":
            # the same chunks with every KDA snapshot as an INT8 record
            self.q8_row = W.state_row_elems(cfg)
            full = [inp.layout.object_bytes(C, g) for g in range(inp.layout.num_object_groups)]
            units = [[(int(j["request"]), int(j["chunk"])) for j in J] for J in inp.jobs]
            inp.object_bytes = [inp.layout.object_bytes_q8(C, self.q8_row, g)
                                for g in range(inp.layout.num_object_groups)]
            self.full_payload = sum(full[g] * len(u) for g, u in enumerate(units))
            inp.jobs, inp.arena_bytes = W.pack_jobs(units, inp.object_bytes)
        if op in ("blocks", "blocks_q8"):
            # the same chunks as block-granular objects holding one KDA
            # snapshot per block (every block boundary of the chunk); with
            # blocks_q8 every snapshot is an INT8 record
            m = C // cfg.N
            units = [[(int(j["request"]), int(j["chunk"]) * m) for j in J] for J in inp.jobs]
            og = range(inp.layout.num_object_groups)
            inp.object_bytes = [inp.layout.object_bytes_blocks(m, True, g) for g in og]
            if op == "blocks_q8":
                self.q8_row = W.state_row_elems(cfg)
                self.full_payload = sum(inp.object_bytes[g] * len(u) for g, u in enumerate(units))
                inp.object_bytes = [inp.layout.object_bytes_blocks_q8(m, True, self.q8_row, g) for g in og]
            inp.jobs, inp.arena_bytes = W.pack_jobs(units, inp.object_bytes)
            self.nb = m
        self.inp, self.L, self.C = inp, inp.layout, C
        L = self.L
        T = torch
        self.main = T.cuda.current_stream(dev)
        self.pool = T.empty(L.pool_bytes, dtype=T.uint8, device=dev)
        W.fill_normal(self.pool, cfg.seed + 101 * rank)
        self.status = T.zeros(1, dtype=T.int32, device=dev)
        self.t_src = [T.from_numpy(t).to(dev) for t in inp.tables_src]
        if cfg.mixed:
            # the load and the store run concurrently on one pool: refuse a
            # batch in which they would touch a common block
            common = lmc.lmc_check_disjoint(L, C, inp.tables_src, inp.load_jobs, inp.tables_src, inp.store_jobs)
            if common >= 0:
                raise RuntimeError(f"mixed step: load and store share block {common}")
            sizes = inp.object_bytes
            self.load_payload = sum(int(sizes[g]) * len(j) for g, j in enumerate(inp.load_jobs))
            self.store_payload = sum(int(sizes[g]) * len(j) for g, j in enumerate(inp.store_jobs))
            self.load_arena = T.empty(inp.load_arena_bytes, dtype=T.uint8, device=dev)
            W.fill_normal(self.load_arena, cfg.seed + 7)
            self.store_arena = T.empty(inp.store_arena_bytes, dtype=T.uint8, device=dev)
            self.load_jobs = [lmc.jobs_to_device(j, dev) for j in inp.load_jobs]
            self.store_jobs = [lmc.jobs_to_device(j, dev) for j in inp.store_jobs]
            self.sa = T.cuda.Stream(dev)
            self.sb = T.cuda.Stream(dev)
            self.chunks = int(sum(len(j) for j in inp.store_jobs) // max(1, L.num_object_groups))
            self.launches_per_step = 2
        else:
            self.load_payload = self.store_payload = inp.payload_bytes
            self.fresh = T.full((L.pool_bytes,), W.SENTINEL, dtype=T.uint8, device=dev)
            self.arena = T.empty(inp.arena_bytes, dtype=T.uint8, device=dev)
            self.t_dst = [T.from_numpy(t).to(dev) for t in inp.tables_dst]
            self.jobs = [lmc.jobs_to_device(j, dev) for j in inp.jobs]
            self.chunks = int(sum(int(x) // C for x in inp.lengths))
            self.launches_per_step = 2
        # every payload byte is read once and written once, by the store and by the load
        self.store_bytes = 2 * self.store_payload
        self.load_bytes = 2 * self.load_payload
        if op in ("q8", "blocks_q8"):
            # the store reads full pages and writes records; the load the reverse
            self.store_bytes = self.load_bytes = self.full_payload + inp.payload_bytes
        self.bytes_per_step = self.store_bytes + self.load_bytes

    def _store(self, pool, tables, jobs):
        lmc = self.lmc
        if self.op == "blocks":
            lmc.lmc_store_blocks(self.L, self.nb, lmc.LMC_KDA_EVERY_BLOCK, pool, tables, jobs, self.arena,
                                 self.status, self.main)
        elif self.op == "blocks_q8":
            lmc.lmc_store_blocks_q8(self.L, self.nb, lmc.LMC_KDA_EVERY_BLOCK, self.q8_row, pool, tables, jobs,
                                    self.arena, self.status, self.main)
        elif self.op == "q8":
            lmc.lmc_store_q8(self.L, self.C, self.q8_row, pool, tables, jobs, self.arena, self.status, self.main)
        else:
            lmc.lmc_store(self.L, self.C, pool, tables, jobs, self.arena, self.status, self.main)

    def _load(self, pool, tables, jobs, stream):
        lmc = self.lmc
        if self.op == "blocks":
            lmc.lmc_load_blocks(self.L, self.nb, lmc.LMC_KDA_EVERY_BLOCK, pool, tables, jobs, self.arena,
                                self.status, stream)
        elif self.op == "blocks_q8":
            lmc.lmc_load_blocks_q8(self.L, self.nb, lmc.LMC_KDA_EVERY_BLOCK, self.q8_row, pool, tables, jobs,
                                   self.arena, self.status, stream)
        elif self.op == "q8":
            lmc.lmc_load_q8(self.L, self.C, self.q8_row, pool, tables, jobs, self.arena, self.status, stream)
        else:
            lmc.lmc_load(self.L, self.C, pool, tables, jobs, self.arena, self.status, stream)

    def new_events(self):
        E = self.torch.cuda.Event
        return [E(enable_timing=True) for _ in range(4)]

    def step(self, ev=None):
        lmc, L, C = self.lmc, self.L, self.C
        if not self.cfg.mixed:
            if ev is not None:
                ev[0].record(self.main)
            self._store(self.pool, self.t_src, self.jobs)
            if ev is not None:
                ev[1].record(self.main)
                ev[2].record(self.main)
            self._load(self.fresh, self.t_dst, self.jobs, self.main)
            if ev is not None:
                ev[3].record(self.main)
            return
        fork = self.torch.cuda.Event()
        fork.record(self.main)
        self.sa.wait_event(fork)
        self.sb.wait_event(fork)
        if ev is not None:
            ev[2].record(self.sa)
            ev[0].record(self.sb)
        lmc.lmc_load(L, C, self.pool, self.t_src, self.load_jobs, self.load_arena, self.status, self.sa)
        lmc.lmc_store(L, C, self.pool, self.t_src, self.store_jobs, self.store_arena, self.status, self.sb)
        if ev is not None:
            ev[3].record(self.sa)
            ev[1].record(self.sb)
        ja, jb = self.torch.cuda.Event(), self.torch.cuda.Event()
        ja.record(self.sa)
        jb.record(self.sb)
        self.main.wait_event(ja)
        self.main.wait_event(jb)

    def setup_e2e(self, parts: int = 64):
        """Pinned host buffers for the end-to-end step: block tables and jobs
        go host -> device each step; objects leave the device for the host
        cache tier (store) and come back from it (load). Plain workloads are
        pipelined over `parts` ranges of (request, chunk) units so that a
        part's device -> host copy overlaps the next part's store and its
        host -> device copy the previous part's load."""
        T, inp = self.torch, self.inp
        pin = lambda a: T.from_numpy(np.ascontiguousarray(a)).pin_memory()
        self.h_tables = [pin(t) for t in inp.tables_src] + ([pin(t) for t in inp.tables_dst] if not self.cfg.mixed else [])
        self.d_tables = self.t_src + ([] if self.cfg.mixed else self.t_dst)
        if self.cfg.mixed:
            self.h_jobs = [pin(j.view(np.uint8)) for j in inp.load_jobs + inp.store_jobs]
            self.d_jobs = self.load_jobs + self.store_jobs
            self._host = [HostArena(T, inp.load_arena_bytes), HostArena(T, inp.store_arena_bytes)]
            self.h_load, self.h_store = self._host[0].tensor, self._host[1].tensor
            self.h_load.copy_(self.load_arena)
            objs_in, objs_out = inp.load_arena_bytes, inp.store_arena_bytes
            self.load_parts = split_parts(inp.load_jobs, inp.object_bytes, parts)
            self.store_parts = split_parts(inp.store_jobs, inp.object_bytes, parts)
            self.s_out = T.cuda.Stream(self.dev)
            self.s_in = T.cuda.Stream(self.dev)
        else:
            self.h_jobs = [pin(j.view(np.uint8)) for j in inp.jobs]
            self.d_jobs = self.jobs
            self._host = [HostArena(T, inp.arena_bytes)]
            self.h_arena = self._host[0].tensor
            objs_in, objs_out = inp.arena_bytes, inp.arena_bytes
            self.parts = split_parts(inp.jobs, inp.object_bytes, parts)
            self.s_out = T.cuda.Stream(self.dev)
            self.s_in = T.cuda.Stream(self.dev)
            self.s_load = T.cuda.Stream(self.dev)
        self.h_status = T.zeros(1, dtype=T.int32, pin_memory=True)
        self.host_memory = "; ".join(h.kind for h in self._host)
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_tables) + \
            sum(j.numel() for j in self.h_jobs) + objs_in
        self.d2h = objs_out + 4

    def close_e2e(self):
        for h in getattr(self, "_host", []):
            h.close()
        self.h_arena = self.h_load = self.h_store = None

    def e2e_step(self):
        lmc, L, C, T = self.lmc, self.L, self.C, self.torch
        for h, d in zip(self.h_tables, self.d_tables):
            d.copy_(h, non_blocking=True)
        for h, d in zip(self.h_jobs, self.d_jobs):
            d.copy_(h, non_blocking=True)
        if self.cfg.mixed:
            # cached objects stream in (host -> device) part by part, each part
            # loaded as it lands; new chunks are stored part by part, each part
            # streamed out (device -> host) as it is written
            ready = T.cuda.Event()
            ready.record(self.main)
            for st in (self.s_in, self.s_out, self.sa, self.sb):
                st.wait_event(ready)
            for rows, lo, hi in self.load_parts:
                jobs = [j[16 * r0:16 * r1] for j, (r0, r1) in zip(self.load_jobs, rows)]
                with T.cuda.stream(self.s_in):
                    self.load_arena[lo:hi].copy_(self.h_load[lo:hi], non_blocking=True)
                    landed = T.cuda.Event()
                    landed.record(self.s_in)
                self.sa.wait_event(landed)
                lmc.lmc_load(L, C, self.pool, self.t_src, jobs, self.load_arena, self.status, self.sa)
            for rows, lo, hi in self.store_parts:
                jobs = [j[16 * r0:16 * r1] for j, (r0, r1) in zip(self.store_jobs, rows)]
                lmc.lmc_store(L, C, self.pool, self.t_src, jobs, self.store_arena, self.status, self.sb)
                written = T.cuda.Event()
                written.record(self.sb)
                with T.cuda.stream(self.s_out):
                    self.s_out.wait_event(written)
                    self.h_store[lo:hi].copy_(self.store_arena[lo:hi], non_blocking=True)
            for st in (self.sa, self.s_out):
                done = T.cuda.Event()
                done.record(st)
                self.main.wait_event(done)
            self.h_status.copy_(self.status, non_blocking=True)
            return
        ready = T.cuda.Event()
        ready.record(self.main)
        self.s_load.wait_event(ready)
        for rows, lo, hi in self.parts:
            jobs = [j[16 * r0:16 * r1] for j, (r0, r1) in zip(self.jobs, rows)]
            self._store(self.pool, self.t_src, jobs)
            stored = T.cuda.Event()
            stored.record(self.main)
            with T.cuda.stream(self.s_out):
                self.s_out.wait_event(stored)
                self.h_arena[lo:hi].copy_(self.arena[lo:hi], non_blocking=True)
                out = T.cuda.Event()
                out.record(self.s_out)
            with T.cuda.stream(self.s_in):
                self.s_in.wait_event(out)
                self.arena[lo:hi].copy_(self.h_arena[lo:hi], non_blocking=True)
                back = T.cuda.Event()
                back.record(self.s_in)
            self.s_load.wait_event(back)
            self._load(self.fresh, self.t_dst, jobs, self.s_load)
        done = T.cuda.Event()
        done.record(self.s_load)
        self.main.wait_event(done)
        self.h_status.copy_(self.status, non_blocking=True)


class CopyStep:
    """In-pool copy-on-write of every KDA snapshot of the batch: one pair per
    (KDA group, request, snapshot) from the batch's block to a spare block of
    a pool twice the batch's size."""

    launches_per_step = 1

    def __init__(self, lmc, torch, cfg, dev, rank, ids):
        self.lmc, self.torch, self.cfg, self.dev = lmc, torch, cfg, dev
        C = lmc.lmc_negotiate_chunk(cfg.requested_chunk, cfg.N)
        build = functools.partial(lmc.lmc_layout_build, cfg.layers, cfg.N, cfg.packed)
        inp = W.make_inputs(cfg, build, C, ids)
        need = inp.layout.num_blocks
        per_block = inp.layout.pool_bytes // need
        self.L = L = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, 2 * need * per_block)
        self.C, self.inp = C, inp
        pairs, nxt, moved = [], need, 0
        for g, kind in enumerate(L.kv_group_kind):
            t = inp.tables_src[g]
            src = t[t >= 0] if kind == "KDA" else np.zeros(0, np.int32)
            pairs.append(np.array([(int(x), nxt + i) for i, x in enumerate(src)],
                                  dtype=lmc.PAIR_DTYPE).reshape(-1))
            nxt += len(src)
            moved += len(src) * sum(L.real_bytes[i] for i in range(L.num_layers) if L.kv_group[i] == g)
        T = torch
        self.main = T.cuda.current_stream(dev)
        self.pool = T.empty(L.pool_bytes, dtype=T.uint8, device=dev)
        W.fill_normal(self.pool, cfg.seed + 101 * rank)
        self.status = T.zeros(1, dtype=T.int32, device=dev)
        self.pairs = [lmc.pairs_to_device(p, dev) for p in pairs]
        self.h_pairs = pairs
        self.store_payload, self.load_payload = moved, 0
        self.store_bytes, self.load_bytes = 2 * moved, 0
        self.bytes_per_step = 2 * moved
        self.chunks = sum(len(p) for p in pairs)

    def new_events(self):
        E = self.torch.cuda.Event
        return [E(enable_timing=True) for _ in range(4)]

    def step(self, ev=None):
        if ev is not None:
            ev[0].record(self.main)
        self.lmc.lmc_copy_blocks(self.L, self.pool, self.pairs, self.h_pairs, self.status, self.main)
        if ev is not None:
            ev[1].record(self.main)
            ev[2].record(self.main)
            ev[3].record(self.main)

    def close_e2e(self):
        pass

    def setup_e2e(self):
        T = self.torch
        self.host_memory = "pinned (cudaHostAlloc)"
        self.h_p = [T.from_numpy(np.ascontiguousarray(p).view(np.uint8)).pin_memory() for p in self.h_pairs]
        self.h_status = T.zeros(1, dtype=T.int32, pin_memory=True)
        self.h2d = sum(p.numel() for p in self.h_p)
        self.d2h = 4

    def e2e_step(self):
        for h, d in zip(self.h_p, self.pairs):
            d.copy_(h, non_blocking=True)
        self.step()
        self.h_status.copy_(self.status, non_blocking=True)


def _capped(cfg, max_chunks, negotiate):
    """The workload with every request cut to at most `max_chunks` whole
    chunks (small cases for profiler captures), or unchanged."""
    if not max_chunks:
        return cfg
    import dataclasses
    C = negotiate(cfg.requested_chunk, cfg.N)
    lengths = tuple(int(min(x, max_chunks * C)) for x in W.request_lengths(cfg))
    return dataclasses.replace(cfg, lengths="fixed", fixed_lengths=lengths)


def _host_link(torch, dev, nbytes=1 << 30, reps=4):
    """The pinned host <-> device link the end-to-end step runs over, measured
    right after it (copy engines, CUDA events): GB/s host to device, device
    to host, and each way with both directions busy."""
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(h2d, d2h):
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for st in (up, down):
            st.wait_event(e0)
        for _ in range(reps):
            if h2d:
                with torch.cuda.stream(up):
                    d_in.copy_(h_in, non_blocking=True)
            if d2h:
                with torch.cuda.stream(down):
                    h_out.copy_(d_out, non_blocking=True)
        for st in (up, down):
            ev = torch.cuda.Event()
            ev.record(st)
            torch.cuda.current_stream(dev).wait_event(ev)
        e1.record()
        torch.cuda.synchronize(dev)
        return round(reps * nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)

    run(True, True)
    out = {"h2d": run(True, False), "d2h": run(False, True), "both_each_way": run(True, True)}
    del h_in, h_out, d_in, d_out
    return out


def _make_step(lmc, torch, cfg, dev, rank, op, n_req):
    ids = list(range(n_req))
    if op == "copy":
        return CopyStep(lmc, torch, cfg, dev, rank, ids)
    return PagingStep(lmc, torch, cfg, dev, rank, ids, op)


def _time_steps(S, torch, dev, dist, local, steps, warmup):
    """W untimed steps, then K steps timed with CUDA events on the launching
    streams, bracketed by a barrier and a device synchronise on both sides;
    SM clocks and throttle reasons sampled during the timed region."""
    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()

    for _ in range(max(warmup, 3)):
        S.step()
    barrier()
    assert int(S.status.item()) == 0, f"device status {int(S.status.item()):#x}"
    evs = [S.new_events() for _ in range(steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        t_start.record(S.main)
        for k in range(steps):
            S.step(evs[k])
        t_end.record(S.main)
        barrier()
    assert int(S.status.item()) == 0
    ms = t_start.elapsed_time(t_end) / steps
    if dist is not None:
        ms = _reduce_max(dist, [ms], dev)[0]
    return {"ms_per_step": ms, "steps": steps, "warmup": max(warmup, 3), "clocks": clk.summary(),
            "store_ms": [e[0].elapsed_time(e[1]) for e in evs], "load_ms": [e[2].elapsed_time(e[3]) for e in evs]}


def _traffic_for(kernels, cfg_index, op):
    """DRAM bytes per launch for the dominant kernel(s), from the committed
    small-case ncu captures scaled to this launch by algorithmic bytes (a
    copy's traffic grows in proportion to the bytes it moves): kernels =
    [(kernel name, algorithmic bytes of this launch)]. None when a capture
    is missing or the kernel source changed since it was taken."""
    total, cases = 0, set()
    for name, nbytes in kernels:
        t = _traffic(name, cfg_index, op)
        if t is None:
            return None, None
        total += t["ratio"] * nbytes
        cases.add(t["case"])
    return int(round(total)), "; ".join(sorted(cases))


def _figures(S, cfg, op, world, t, peak, peak_src):
    """Throughput, per-kernel times and the roofline of the dominant kernel
    for one timed workload."""
    ms = t["ms_per_step"]
    value = S.bytes_per_step * world / (ms * 1e-3) / 1e9
    st_avg, ld_avg = statistics.mean(t["store_ms"]), statistics.mean(t["load_ms"])
    suffix = "_q8_kernel" if op in ("q8", "blocks_q8") else "_kernel"
    if op == "copy":
        dominant, dom_bytes, dom_ms = "lmc_copy_kernel", S.bytes_per_step, st_avg
        parts = [("lmc_copy_kernel", dom_bytes)]
    elif cfg.mixed:
        # the two kernels share HBM concurrently: the roofline is the step's
        dominant, dom_bytes, dom_ms = "lmc_store_kernel+lmc_load_kernel (concurrent)", S.bytes_per_step, ms
        parts = [("lmc_store_kernel", S.store_bytes), ("lmc_load_kernel", S.load_bytes)]
    elif st_avg >= ld_avg:
        dominant, dom_bytes, dom_ms = "lmc_store" + suffix, S.store_bytes, st_avg
        parts = [(dominant, dom_bytes)]
    else:
        dominant, dom_bytes, dom_ms = "lmc_load" + suffix, S.load_bytes, ld_avg
        parts = [(dominant, dom_bytes)]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic, source = _traffic_for(parts, cfg.index, op)
    return {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms, 4), "steps": t["steps"],
        "warmup": t["warmup"],
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "pct_of_nominal_hbm": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "chunks_per_s": round(S.chunks * world / (ms * 1e-3), 1),
        "store": _with_frac(_kernel_times(S.store_bytes, t["store_ms"]), peak),
        "load": _with_frac(_kernel_times(S.load_bytes, t["load_ms"]), peak),
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 2), "peak": peak,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs: copy read+write)",
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "traffic_source": (f"ncu dram__bytes_read.sum + dram__bytes_write.sum per launch on a small case "
                                        f"({source}), scaled to this launch by algorithmic bytes") if source else None,
                     "algorithmic_bytes_per_launch": dom_bytes},
        "clocks": t["clocks"],
    }


# Further lines of the default run: the other workloads and operations, each
# timed on its own in the same process (K capped to keep the run short).
EXTRA_LINES = [("per_config", 2, "paging", 50), ("per_config", 3, "paging", 10), ("per_config", 4, "paging", 10),
               ("per_op", 1, "q8", 50), ("per_op", 3, "q8", 10), ("per_op", 2, "blocks", 50),
               ("per_op", 2, "blocks_q8", 50), ("per_op", 1, "copy", 50)]


def run_gpu(args):
    import torch

    import state_cache_paging_gb300 as lmc

    dist, rank, world, local = _dist()
    if dist is not None:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = _capped(W.CONFIGS[args.config], args.max_chunks, lmc.lmc_negotiate_chunk)
    n_req = _step_requests(cfg, args.requests)
    peak, peak_src = _peaks()
    # each rank runs its own independent copy of the batch (weak scaling)
    S = _make_step(lmc, torch, cfg, dev, rank, args.op, n_req)
    L = S.L
    t = _time_steps(S, torch, dev, dist, local, args.steps, args.warmup)

    # the end-to-end step needs the objects in pinned host memory; if any rank
    # cannot pin them, every rank skips it (the ranks agree before going on)
    e2e_err = None
    try:
        if args.op == "copy":
            S.setup_e2e()
        else:
            S.setup_e2e(args.e2e_parts)
    except (RuntimeError, MemoryError) as err:
        e2e_err = f"{type(err).__name__}: {err}".splitlines()[0][:200]
    e2e_ok = _all_ranks(dist, e2e_err is None, dev)
    e2e_ms = 0.0
    if e2e_ok:
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        for _ in range(2):
            S.e2e_step()
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(S.main)
        for _ in range(e2e_steps):
            S.e2e_step()
        e1.record(S.main)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        assert int(S.h_status.item()) == 0
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
        if dist is not None:
            e2e_ms = _reduce_max(dist, [e2e_ms], dev)[0]
        link = _host_link(torch, dev)

    fig = _figures(S, cfg, args.op, world, t, peak, peak_src)
    line = {
        "metric": METRIC, "value": fig["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": fig["warmup"], "ms_per_step": fig["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": dict(_workload_config(cfg, args.op, n_req, S.store_payload, S.load_payload, S.C, L.pool_bytes,
                                        world), **({"max_chunks": args.max_chunks} if args.max_chunks else {})),
        **{k: fig[k] for k in ("pct_of_hbm_peak", "pct_of_nominal_hbm", "chunks_per_s", "store", "load", "roofline")},
        "e2e": ({"value": round(S.bytes_per_step * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                 "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": S.h2d, "d2h_bytes_per_step": S.d2h,
                 "parts": None if args.op == "copy" else args.e2e_parts,
                 "host_memory": S.host_memory, "host_link_gbs": link} if e2e_ok else
                {"value": None, "unit": "GB/s", "unavailable": e2e_err or "a rank could not pin its host buffers"}),
        "gpu_launches": S.launches_per_step * args.steps,
        "clocks": fig["clocks"],
    }
    if world == 1 and not args.no_cpu_baseline and args.op == "paging":
        threads = os.cpu_count() or 1
        # the oracle on the same payload as the step, on every host core
        # (about 10-15 s of passes), then on one core (two passes); the pool is
        # this step's own device pool, copied to the host
        pool_of = lambda inp: S.pool.cpu().numpy()  # noqa: E731
        res = oracle_time(args.config, n_req, threads, seconds=15.0, pool_of=pool_of)
        one = oracle_time(args.config, n_req, 1, reps=2, pool_of=pool_of)
        line["cpu_baseline"] = {k: res[k] for k in ("value", "unit", "cores", "kind", "sample", "chunks_per_s",
                                                   "seconds", "waves")}
        line["cpu_baseline"]["same_payload_as_step"] = res["payload_bytes_per_pass"] == \
            S.store_payload + S.load_payload
        line["cpu_baseline"]["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}
    if e2e_ok:
        S.close_e2e()
    del S
    torch.cuda.empty_cache()

    if args.extra_lines:
        # the other workloads and operations, so that one default run covers
        # every line; each is built, timed and freed in turn
        for key, idx, op, k_cap in EXTRA_LINES:
            if (idx, op) == (args.config, args.op):
                continue
            c = W.CONFIGS[idx]
            nr = _step_requests(c)
            S = _make_step(lmc, torch, c, dev, rank, op, nr)
            tt = _time_steps(S, torch, dev, dist, local, min(args.steps, k_cap), args.warmup)
            f = _figures(S, c, op, world, tt, peak, peak_src)
            entry = {"config": _workload_config(c, op, nr, S.store_payload, S.load_payload, S.C, S.L.pool_bytes,
                                                world), **f, "gpu_launches": S.launches_per_step * tt["steps"]}
            line.setdefault(key, {})[f"config{idx}" + ("" if op == "paging" else f"/{op}")] = entry
            del S
            torch.cuda.empty_cache()
        line["gpu_launches"] += sum(e["gpu_launches"] for key in ("per_config", "per_op")
                                    for e in line.get(key, {}).values())
    if rank == 0:
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
    ap.add_argument("--max-chunks", type=int, default=None,
                    help="cut every request to at most K whole chunks (small cases for profiler captures)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-parts", type=int, default=64,
                    help="ranges of (request, chunk) units the end-to-end step is pipelined over")
    ap.add_argument("--impl", choices=["lmc", "reference"], default="lmc")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-lines", dest="extra_lines", action="store_false",
                    help="time only the selected workload (the default run also times configs 2-4 and the "
                         "codec, block and copy operations, each as its own entry)")
    ap.add_argument("--op", choices=["paging", "blocks", "copy", "q8", "blocks_q8"], default="paging",
                    help="paging: store + load by chunk; blocks: block-granular objects with one KDA "
                         "snapshot per block; copy: in-pool copy of every KDA snapshot; q8: store + load "
                         "with KDA snapshots as INT8 records; blocks_q8: block-granular objects with every "
                         "snapshot as an INT8 record")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

"""Helpers for the GPU parity tests: device inputs for a workload, calls
through the C ABI, and oracle checks that scale to full-size workloads
(every object and every loaded page compared, streamed in slices).

Inputs come from the seeded generators (workloads/) using the ORACLE's
layout; the library's layout is asserted equal before anything runs, so the
two sides see the same pools, tables and jobs. Expected values come only from
the oracle.
"""
from __future__ import annotations

import functools
import mmap

import numpy as np
import torch

import oracle
import workloads as W
import state_cache_paging_gb300 as lmc

LAYOUT_FIELDS = ("num_kv_groups", "num_object_groups", "num_slabs", "page_size", "block_stride",
                 "num_blocks", "pool_bytes", "kv_group", "slot", "object_group", "kv_group_kind",
                 "kv_group_size", "real_bytes", "page_bytes", "base", "stride", "kinds")


def negotiated(cfg):
    C = oracle.negotiate_chunk(cfg.requested_chunk, cfg.N)
    assert lmc.lmc_negotiate_chunk(cfg.requested_chunk, cfg.N) == C
    return C


def case_inputs(cfg, request_ids=None, split=True, separate=True):
    """(inputs built on the oracle's layout, the library's equal layout)."""
    C = negotiated(cfg)
    inp = W.make_inputs(cfg, functools.partial(oracle.layout, cfg.layers, cfg.N, cfg.packed,
                                               split_groups=split, separate_object_groups=separate),
                        C, request_ids)
    Lo = inp.layout
    Lp = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, Lo.pool_bytes, split, separate)
    for f in LAYOUT_FIELDS:
        assert getattr(Lp, f) == getattr(Lo, f), f
    for g in range(Lo.num_object_groups):
        assert Lp.object_bytes(C, g) == Lo.object_bytes(C, g)
    return inp, Lp


def dev_tables(tables, dev):
    return [torch.from_numpy(np.ascontiguousarray(t)).to(dev) for t in tables]


def dev_jobs(jobs, dev):
    return [lmc.jobs_to_device(j, dev) for j in jobs]


def object_span(inp, og, job):
    off = int(job["offset"])
    return off, off + int(inp.object_bytes[og])


# ---------------------------------------------------------------------------
# Full-size comparison with the oracle, streamed in arena-ordered slices so
# the host holds a few GB whatever the pool's size
# ---------------------------------------------------------------------------

SLICE_BYTES = 2 << 30
ARENA_FILL = 0x3C  # arenas start filled with this byte on both sides


class LazyHost:
    """n bytes of private anonymous host memory standing for a pool on the
    oracle's side: a page costs memory only once written, and release()
    hands every page back (all bytes read as zero again)."""

    def __init__(self, n):
        self.n = int(n)
        self._map = mmap.mmap(-1, max(self.n, 1), flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        self.a = np.frombuffer(self._map, dtype=np.uint8, count=self.n)

    def release(self):
        self._map.madvise(mmap.MADV_DONTNEED)


def fetch(dev_buf, lo, hi, out=None):
    """Device bytes [lo, hi) copied into `out` (a numpy view) or a new array."""
    if out is None:
        out = np.empty(hi - lo, dtype=np.uint8)
    torch.from_numpy(out).copy_(dev_buf[lo:hi])
    return out


def job_slices(jobs, sizes, limit=None):
    """Every job of every object group in arena order, cut into runs whose
    objects span at most ~limit bytes (default SLICE_BYTES): yields
    (per-group job subsets, lo, hi) where [lo, hi) is the run's arena range."""
    limit = SLICE_BYTES if limit is None else limit
    order = sorted((int(j["offset"]), g, k) for g, J in enumerate(jobs) for k, j in enumerate(J))
    start = 0
    while start < len(order):
        lo = order[start][0]
        end = start
        hi = lo
        while end < len(order):
            off, g, _ = order[end]
            stop = off + int(sizes[g])
            if end > start and stop - lo > limit:
                break
            hi = max(hi, stop)
            end += 1
        picks = [[] for _ in jobs]
        for _, g, k in order[start:end]:
            picks[g].append(k)
        yield [J[np.array(p, dtype=np.int64)] for J, p in zip(jobs, picks)], lo, hi
        start = end


def _rebased(sel, lo):
    out = []
    for J in sel:
        J = J.copy()
        J["offset"] -= lo
        out.append(J)
    return out


def _first_diff(got, want, base):
    bad = np.flatnonzero(got != want)
    return f"{bad.size} bytes differ, first at {base + int(bad[0])}"


def check_store_streamed(Lo, C, pool_dev, arena_dev, jobs, sizes, tables, oracle_store, nb=0, kda_every=False,
                         fill=ARENA_FILL):
    """Every object of `jobs` is recomputed by the oracle (oracle_store(pool,
    tables, jobs, arena) -> status) from the pool pages it reads, fetched from
    the device, and compared byte for byte with the device arena (filled with
    `fill` before the store, like the oracle's). Returns the object bytes
    compared, which a test sets against the full payload."""
    host = LazyHost(Lo.pool_bytes)
    checked = 0
    for sel, lo, hi in job_slices(jobs, sizes):
        pages, st = oracle.list_pages(Lo, C, tables, sel, 1 << 62, nb=nb, kda_every=kda_every)
        assert st == 0
        for po, n in zip(pages["pool_offset"].tolist(), pages["bytes"].tolist()):
            fetch(pool_dev, po, po + n, host.a[po:po + n])
        want = np.full(hi - lo, fill, dtype=np.uint8)
        assert oracle_store(host.a, tables, _rebased(sel, lo), want) == 0
        got = fetch(arena_dev, lo, hi)
        if not np.array_equal(got, want):
            raise AssertionError("store: " + _first_diff(got, want, lo))
        checked += sum(int(sizes[g]) * len(J) for g, J in enumerate(sel))
        host.release()
    return checked


def check_load_streamed(Lo, C, dest_dev, arena_dev, jobs, sizes, tables, oracle_load, nb=0, kda_every=False):
    """The oracle (oracle_load(pool, tables, jobs, arena) -> status) scatters
    every object of `jobs`, read from the device arena, and every page it
    writes is compared byte for byte with the device pool. Returns the page
    bytes compared."""
    host = LazyHost(Lo.pool_bytes)
    checked = 0
    for sel, lo, hi in job_slices(jobs, sizes):
        src = fetch(arena_dev, lo, hi)
        assert oracle_load(host.a, tables, _rebased(sel, lo), src) == 0
        pages, st = oracle.list_pages(Lo, C, tables, sel, 1 << 62, nb=nb, kda_every=kda_every)
        assert st == 0
        for po, n in zip(pages["pool_offset"].tolist(), pages["bytes"].tolist()):
            got = fetch(dest_dev, po, po + n)
            if not np.array_equal(got, host.a[po:po + n]):
                raise AssertionError("load: " + _first_diff(got, host.a[po:po + n], po))
            checked += n
        host.release()
    return checked


def check_untouched(inp, pool_dev, jobs, tables, arena_bytes, fill_value):
    """Every pool byte outside the pages the oracle names still holds
    `fill_value` (checked on the device, any size)."""
    Lo, C = inp.layout, inp.C
    pages, st = oracle.list_pages(Lo, C, tables, jobs, arena_bytes)
    assert st == 0
    ref = torch.full_like(pool_dev, fill_value)
    for pg in pages:
        lo, n = int(pg["pool_offset"]), int(pg["bytes"])
        ref[lo:lo + n] = pool_dev[lo:lo + n]
    ok = torch.equal(ref, pool_dev)
    del ref
    return ok

"""Helpers for the GPU parity tests: device inputs for a workload, calls
through the C ABI, and oracle checks that scale to full-size workloads.

Inputs come from the seeded generators (workloads/) using the ORACLE's
layout; the library's layout is asserted equal before anything runs, so the
two sides see the same pools, tables and jobs. Expected values come only from
the oracle.
"""
from __future__ import annotations

import functools

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


def pick_jobs(jobs, per_group, rng):
    out = []
    for J in jobs:
        k = min(per_group, len(J))
        idx = np.sort(rng.choice(len(J), size=k, replace=False)) if k else np.zeros(0, dtype=np.int64)
        out.append(J[idx])
    return out


def _fetch(dev_buf, lo, hi):
    return dev_buf[lo:hi].cpu().numpy()


def check_store_sampled(inp, pool_dev, arena_dev, jobs, tables, arena_bytes, per_group, rng):
    """The oracle recomputes a sample of objects from the pages it names and
    the bytes are compared with the library's objects."""
    Lo, C = inp.layout, inp.C
    sel = pick_jobs(jobs, per_group, rng)
    pages, st = oracle.list_pages(Lo, C, tables, sel, arena_bytes)
    assert st == 0
    host_pool = np.zeros(Lo.pool_bytes, dtype=np.uint8)  # pages mapped lazily
    for pg in pages:
        lo, n = int(pg["pool_offset"]), int(pg["bytes"])
        host_pool[lo:lo + n] = _fetch(pool_dev, lo, lo + n)
    arena_o = np.zeros(arena_bytes, dtype=np.uint8)
    assert oracle.store(Lo, C, host_pool, tables, sel, arena_o) == 0
    n_checked = 0
    for og, J in enumerate(sel):
        for job in J:
            lo, hi = object_span(inp, og, job)
            assert np.array_equal(_fetch(arena_dev, lo, hi), arena_o[lo:hi]), (og, job)
            n_checked += hi - lo
    return n_checked


def check_load_sampled(inp, pool_dev, arena_dev, jobs, tables, arena_bytes, per_group, rng):
    """The oracle scatters a sample of objects; every page it writes is
    compared with the library's pool."""
    Lo, C = inp.layout, inp.C
    sel = pick_jobs(jobs, per_group, rng)
    host_arena = np.zeros(arena_bytes, dtype=np.uint8)
    for og, J in enumerate(sel):
        for job in J:
            lo, hi = object_span(inp, og, job)
            host_arena[lo:hi] = _fetch(arena_dev, lo, hi)
    host_pool = np.zeros(Lo.pool_bytes, dtype=np.uint8)
    assert oracle.load(Lo, C, host_pool, tables, sel, host_arena) == 0
    pages, st = oracle.list_pages(Lo, C, tables, sel, arena_bytes)
    assert st == 0
    n_checked = 0
    for pg in pages:
        lo, n = int(pg["pool_offset"]), int(pg["bytes"])
        assert np.array_equal(_fetch(pool_dev, lo, lo + n), host_pool[lo:lo + n]), pg
        n_checked += n
    return n_checked


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

"""The streamed full-size checker of the GPU tests, run on the CPU with
host tensors standing in for device buffers: it must compare every byte of
both directions and catch a single wrong byte anywhere."""
import numpy as np
import pytest
import torch

import gpu_harness as H
import oracle
import workloads as W


@pytest.fixture
def small_slices(monkeypatch):
    monkeypatch.setattr(H, "SLICE_BYTES", 300_000)  # several slices on the tiny workload


def _tiny():
    cfg = W.CONFIGS[0]
    inp, _ = H.case_inputs(cfg)
    Lo, C = inp.layout, inp.C
    pool_h = W.fill_normal_np(Lo.pool_bytes, 5)
    arena = np.full(inp.arena_bytes, H.ARENA_FILL, dtype=np.uint8)
    assert oracle.store(Lo, C, pool_h, inp.tables_src, inp.jobs, arena) == 0
    fresh = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
    assert oracle.load(Lo, C, fresh, inp.tables_dst, inp.jobs, arena) == 0
    return inp, torch.from_numpy(pool_h), torch.from_numpy(arena), torch.from_numpy(fresh)


def _calls(Lo, C):
    return (lambda p, t, j, a: oracle.store(Lo, C, p, t, j, a), lambda p, t, j, a: oracle.load(Lo, C, p, t, j, a))


def test_slices_cover_every_job_once(small_slices):
    inp, *_ = _tiny()
    seen = [[] for _ in inp.jobs]
    ranges = []
    for sel, lo, hi in H.job_slices(inp.jobs, inp.object_bytes):
        ranges.append((lo, hi))
        for g, J in enumerate(sel):
            seen[g] += [int(x) for x in J["offset"]]
            assert all(lo <= int(o) and int(o) + inp.object_bytes[g] <= hi for o in J["offset"])
    assert len(ranges) > 3
    assert all(a[1] <= b[0] for a, b in zip(ranges, ranges[1:]))
    for g, J in enumerate(inp.jobs):
        assert sorted(seen[g]) == sorted(int(x) for x in J["offset"])


def test_streamed_checks_count_the_full_payload(small_slices):
    inp, pool, arena, fresh = _tiny()
    Lo, C = inp.layout, inp.C
    st, ld = _calls(Lo, C)
    assert H.check_store_streamed(Lo, C, pool, arena, inp.jobs, inp.object_bytes, inp.tables_src, st) \
        == inp.payload_bytes
    assert H.check_load_streamed(Lo, C, fresh, arena, inp.jobs, inp.object_bytes, inp.tables_dst, ld) \
        == inp.payload_bytes


@pytest.mark.parametrize("where", [0, 0.37, 0.999])
def test_streamed_checks_catch_one_wrong_byte(small_slices, where):
    inp, pool, arena, fresh = _tiny()
    Lo, C = inp.layout, inp.C
    st, ld = _calls(Lo, C)
    k = int(where * (inp.arena_bytes - 1))
    arena[k] ^= 1
    with pytest.raises(AssertionError, match="store"):
        H.check_store_streamed(Lo, C, pool, arena, inp.jobs, inp.object_bytes, inp.tables_src, st)
    arena[k] ^= 1
    pages, _ = oracle.list_pages(Lo, C, inp.tables_dst, inp.jobs, inp.arena_bytes)
    pg = pages[int(where * (len(pages) - 1))]
    b = int(pg["pool_offset"]) + int(where * (int(pg["bytes"]) - 1))
    fresh[b] ^= 0x80
    with pytest.raises(AssertionError, match="load"):
        H.check_load_streamed(Lo, C, fresh, arena, inp.jobs, inp.object_bytes, inp.tables_dst, ld)

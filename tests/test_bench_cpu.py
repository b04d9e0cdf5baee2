"""Host logic of the benchmark's end-to-end pipeline (no GPU): the parts a
step is split into cover every job once and map to disjoint arena ranges."""
import functools
import os
import sys

import numpy as np
import pytest

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("cfg_index,ids", [(0, None), (1, None), (2, None), (3, [1]), (4, list(range(40)))])
@pytest.mark.parametrize("parts", [1, 3, 16])
def test_split_parts_cover_jobs_once(cfg_index, ids, parts):
    cfg = W.CONFIGS[cfg_index]
    C = oracle.negotiate_chunk(cfg.requested_chunk, cfg.N)
    inp = W.make_inputs(cfg, functools.partial(oracle.layout, cfg.layers, cfg.N, cfg.packed), C, ids)
    sets = [(inp.load_jobs, inp.load_arena_bytes), (inp.store_jobs, inp.store_arena_bytes)] if cfg.mixed \
        else [(inp.jobs, inp.arena_bytes)]
    for jobs, nbytes in sets:
        out = bench.split_parts(jobs, inp.object_bytes, parts)
        assert 1 <= len(out) <= parts
        seen = [np.zeros(len(J), dtype=np.int8) for J in jobs]
        for rows, lo, hi in out:
            for g, (r0, r1) in enumerate(rows):
                seen[g][r0:r1] += 1
                offs = jobs[g]["offset"][r0:r1].astype(np.int64)
                assert (offs >= lo).all() and (offs + inp.object_bytes[g] <= hi).all()
        assert all((x == 1).all() for x in seen)
        # the parts' arena ranges tile [0, arena bytes) without overlap
        spans = sorted((lo, hi) for _, lo, hi in out)
        assert spans[0][0] == 0 and spans[-1][1] == nbytes
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))

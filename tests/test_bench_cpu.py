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


def test_mixed_step_load_and_store_blocks_are_disjoint(lmc):
    """The mixed workload's load (cached chunks) and store (new chunks) touch
    disjoint blocks, so the two streams never race (the library's guard the
    benchmark calls); a batch whose store repeats a loaded chunk shares a
    block."""
    cfg = W.CONFIGS[4]
    C = oracle.negotiate_chunk(cfg.requested_chunk, cfg.N)
    inp = W.make_inputs(cfg, functools.partial(oracle.layout, cfg.layers, cfg.N, cfg.packed), C, list(range(40)))
    L = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, inp.layout.pool_bytes)
    T = inp.tables_src
    assert sum(len(j) for j in inp.load_jobs) and sum(len(j) for j in inp.store_jobs)
    assert lmc.lmc_check_disjoint(L, C, T, inp.load_jobs, T, inp.store_jobs) == -1
    bad = [J.copy() for J in inp.store_jobs]
    g = next(g for g, J in enumerate(inp.load_jobs) if len(J))
    bad[g] = np.concatenate([bad[g], inp.load_jobs[g][:1]])
    assert lmc.lmc_check_disjoint(L, C, T, inp.load_jobs, T, bad) >= 0


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle timed on the host cores) prints
    one JSON line with the benchmark contract's keys."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "0",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


def test_kernel_times_mean_median_best():
    t = bench._kernel_times(2_000_000_000, [2.0, 1.0, 4.0])
    assert t["ms"] == round(7 / 3, 4) and t["median_ms"] == 2.0 and t["best_ms"] == 1.0
    assert t["best_gbs"] == 2000.0 and t["median_gbs"] == 1000.0
    assert bench._kernel_times(0, [0.002])["gbs"] is None and t["bytes"] == 2_000_000_000


def test_reference_arm_times_the_whole_step_payload():
    """The oracle arm moves the GPU step's whole payload (both directions of
    config 0: 2,147,328 object bytes each), and its `config` carries the
    same workload keys as the GPU line."""
    res = bench.oracle_time(0, 2, threads=2, reps=1, warmup=1)
    c = res["config"]
    assert res["payload_bytes_per_pass"] == 2 * 2_147_328
    assert c["store_payload_bytes"] == c["load_payload_bytes"] == 2_147_328
    assert c["requests"] == 2 and c["chunk"] == 128 and c["N"] == 64 and c["layout"] == "padded"
    assert c["pool_bytes"] == 64 * 73_728 and res["waves"] == 1
    assert set(c) == {"workload", "index", "op", "requests", "scope", "store_payload_bytes", "load_payload_bytes",
                      "chunk", "N", "layout", "pool_bytes", "l2", "parallelism"}


def test_reference_arm_runs_in_waves_when_host_memory_is_short(monkeypatch):
    """With too little host memory for one pass, the requests run in waves
    and the payload moved is unchanged."""
    monkeypatch.setattr(bench, "_host_free_bytes", lambda: 16 << 20)
    res = bench.oracle_time(0, 2, threads=1, reps=1, warmup=1)
    assert res["waves"] == 2 and res["payload_bytes_per_pass"] == 2 * 2_147_328


def test_step_requests_one_wave_of_k3():
    assert bench._step_requests(W.CONFIGS[3]) == 1
    assert bench._step_requests(W.CONFIGS[1]) == 32 and bench._step_requests(W.CONFIGS[1], 4) == 4


def test_capped_requests_for_small_captures():
    import state_cache_paging_gb300 as lmc
    c = bench._capped(W.CONFIGS[3], 4, lmc.lmc_negotiate_chunk)
    assert c.fixed_lengths == (4 * 1536,) * 4 and c.index == 3
    assert bench._capped(W.CONFIGS[1], None, lmc.lmc_negotiate_chunk) is W.CONFIGS[1]


def test_each_kernel_reports_its_fraction_of_peak():
    t = bench._with_frac(bench._kernel_times(7_000_000_000, [1.0]), 7000.0)
    assert t["gbs"] == 7000.0 and t["frac_of_peak"] == 1.0
    assert bench._with_frac(bench._kernel_times(0, [1.0]), 7000.0)["frac_of_peak"] is None


def test_host_arena_refuses_more_than_free_memory(monkeypatch):
    """The end-to-end step's host arena checks free host memory before it
    faults pages in, and raises MemoryError (the step then reports itself
    unavailable) rather than risk running the host out of memory."""
    import torch
    monkeypatch.setattr(bench, "_host_free_bytes", lambda: 1 << 20)
    with pytest.raises(MemoryError):
        bench.HostArena(torch, 1 << 30)

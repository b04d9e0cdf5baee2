"""GPU parity: liblmc's store and load against the CPU oracle, byte for byte.

Small cases (the tiny workload, random specs, every error path) are compared
in full. The full-size workloads run in the launch configuration the
benchmark times, and every object and every loaded page is compared with the
oracle too, streamed through host memory in slices (each test asserts that
the bytes compared equal the full payload of each direction); pool bytes
outside the addressed pages are checked untouched on the device.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import oracle_pins as P
import workloads as W
from gpu_harness import (ARENA_FILL, LazyHost, case_inputs, check_load_streamed, check_store_streamed,
                         check_untouched, dev_jobs, dev_tables, fetch)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _full_exact(lmc, inp, Lp, pool_offset=0, arena_offset=0):
    """Store + load of every job, compared in full with the oracle."""
    Lo, C = inp.layout, inp.C
    pool_h = W.fill_normal_np(Lo.pool_bytes, inp.cfg.seed + 17)
    buf = torch.empty(Lo.pool_bytes + 64, dtype=torch.uint8, device=DEV)
    pool = buf[pool_offset:pool_offset + Lo.pool_bytes]
    pool.copy_(torch.from_numpy(pool_h))
    abuf = torch.full((inp.arena_bytes + 64,), 0x3C, dtype=torch.uint8, device=DEV)
    arena = abuf[arena_offset:arena_offset + inp.arena_bytes]
    fbuf = torch.full((Lo.pool_bytes + 64,), W.SENTINEL, dtype=torch.uint8, device=DEV)
    fresh = fbuf[pool_offset:pool_offset + Lo.pool_bytes]
    st = _status()
    jobs = dev_jobs(inp.jobs, DEV)
    lmc.lmc_store(Lp, C, pool, dev_tables(inp.tables_src, DEV), jobs, arena, st)
    lmc.lmc_load(Lp, C, fresh, dev_tables(inp.tables_dst, DEV), jobs, arena, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    arena_o = np.full(inp.arena_bytes, 0x3C, dtype=np.uint8)
    assert oracle.store(Lo, C, pool_h, inp.tables_src, inp.jobs, arena_o) == 0
    fresh_o = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
    assert oracle.load(Lo, C, fresh_o, inp.tables_dst, inp.jobs, arena_o) == 0
    assert np.array_equal(arena.cpu().numpy(), arena_o)
    assert np.array_equal(fresh.cpu().numpy(), fresh_o)
    # guard bytes around the buffers are untouched
    assert (abuf[:arena_offset] == 0x3C).all() and (abuf[arena_offset + inp.arena_bytes:] == 0x3C).all()
    assert (fbuf[:pool_offset] == W.SENTINEL).all() and (fbuf[pool_offset + Lo.pool_bytes:] == W.SENTINEL).all()


def test_tiny_workload_exact(lmc):
    inp, Lp = case_inputs(W.CONFIGS[0])
    _full_exact(lmc, inp, Lp)


@pytest.mark.parametrize("pool_offset,arena_offset", [(0, 0), (8, 0), (0, 4), (3, 5)])
def test_tiny_workload_unaligned_buffers(lmc, pool_offset, arena_offset):
    """Buffers that are not 16-byte aligned take the byte-wise path."""
    inp, Lp = case_inputs(W.CONFIGS[0])
    _full_exact(lmc, inp, Lp, pool_offset, arena_offset)


def _random_cfg(rng, t):
    spec = P.random_spec(rng, int(rng.integers(2, 9)))
    spec[0] = W.mla(int(rng.choice([16, 32, 48, 1152])))
    spec[-1] = W.kda(int(rng.choice([8, 64, 768])), 3, int(rng.choice([1, 2, 4])), int(rng.choice([8, 16, 64])))
    N = int(rng.choice([2, 4, 16, 64]))
    lengths = tuple(int(x) for x in rng.integers(N, 40 * N, size=int(rng.integers(1, 6))))
    return W.Config(100 + t, "random", spec, N=N, requested_chunk=int(rng.integers(0, 5 * N)),
                    packed=bool(t % 2), num_requests=len(lengths), lengths="fixed",
                    fixed_lengths=lengths, snapshot=("block" if t % 3 else "chunk"), seed=t)


@pytest.mark.parametrize("t", range(24))
def test_random_specs_exact(lmc, t):
    rng = np.random.default_rng(1000 + t)
    cfg = _random_cfg(rng, t)
    inp, Lp = case_inputs(cfg, split=bool((t // 2) % 2), separate=bool((t // 4) % 2 == 0))
    _full_exact(lmc, inp, Lp)


def test_odd_page_sizes_exact(lmc):
    """Pages that are not 16-byte multiples (byte-wise path, ragged tiles)."""
    spec = [W.mla(18), {"kind": "KDA", "token_bytes": 0, "conv_bytes": 6, "rec_bytes": 70001, "window": 0},
            W.swa(7, 32), W.mla(18)]
    cfg = W.Config(200, "odd", spec, N=8, requested_chunk=20, packed=True, num_requests=3,
                   lengths="fixed", fixed_lengths=(50, 97, 33), seed=5)
    inp, Lp = case_inputs(cfg)
    _full_exact(lmc, inp, Lp)


def test_large_pages_exact(lmc):
    """Pages far larger than one tile (a 33 MB KDA state, 1.2 MB MLA page)."""
    spec = [W.kda(3 * 64 * 128, 3, 128, 256), W.mla(1152), W.kda(3 * 64 * 128, 3, 128, 256)]
    cfg = W.Config(201, "large", spec, N=1024, requested_chunk=2000, packed=False, num_requests=2,
                   lengths="fixed", fixed_lengths=(4100, 6200), seed=6)
    inp, Lp = case_inputs(cfg)
    _full_exact(lmc, inp, Lp)


@pytest.mark.parametrize("packed", [False, True])
def test_step_boundary_snapshots_exact(lmc, packed):
    """The >= 2N scheduler regime ("Kimi-Linear" recipe, Why these settings:
    one scheduler step covers more than one block, and the KDA state is
    saved only where the step ends): with C = N and steps of 3 blocks, the KDA tables hold states
    only at positions 3k + 2. With separate object groups the caller stores
    every chunk's MLA object and only the step-end chunks' KDA objects: exact
    against the oracle. A KDA object asked for at a chunk inside a step finds
    no snapshot: NO_SNAPSHOT, its pages skipped, the same as the oracle."""
    spec = [W.kda(48, 3, 2, 32), W.kda(48, 3, 2, 32), W.kda(48, 3, 2, 32), W.mla(64)]
    cfg = W.Config(230 + int(packed), "steps", spec, N=16, requested_chunk=16, packed=packed, num_requests=3,
                   lengths="fixed", fixed_lengths=(150, 97, 200), seed=23)
    inp, Lp = case_inputs(cfg)
    Lo, C = inp.layout, inp.C
    assert C == cfg.N
    kda_groups = [k for k, kind in enumerate(Lo.kv_group_kind) if kind == "KDA"]
    for tables in (inp.tables_src, inp.tables_dst):
        for k in kda_groups:
            t = tables[k]
            cols = np.arange(t.shape[1])
            t[:, (cols + 1) % 3 != 0] = -1  # states only where a step of 3 blocks ended
    og_kda = Lo.object_group[Lo.kinds.index("KDA")]
    step_end = (inp.jobs[og_kda]["chunk"] + 1) % 3 == 0
    inside = inp.jobs[og_kda][~step_end][:1].copy()
    units = [[(int(j["request"]), int(j["chunk"])) for j in J] for J in inp.jobs]
    units[og_kda] = [(int(j["request"]), int(j["chunk"])) for j in inp.jobs[og_kda][step_end]]
    assert units[og_kda] and inside.size
    inp.jobs, inp.arena_bytes = W.pack_jobs(units, inp.object_bytes)
    _full_exact(lmc, inp, Lp)
    # one KDA object inside a step: no snapshot there
    jobs = [J.copy() for J in inp.jobs]
    inside["offset"] = inp.arena_bytes
    jobs[og_kda] = np.concatenate([jobs[og_kda], inside])
    nbytes = inp.arena_bytes + inp.object_bytes[og_kda]
    pool_h = W.fill_normal_np(Lo.pool_bytes, 29)
    arena = torch.full((nbytes,), 0x3C, dtype=torch.uint8, device=DEV)
    st = _status()
    lmc.lmc_store(Lp, C, torch.from_numpy(pool_h).to(DEV), dev_tables(inp.tables_src, DEV), dev_jobs(jobs, DEV),
                  arena, st)
    torch.cuda.synchronize()
    arena_o = np.full(nbytes, 0x3C, dtype=np.uint8)
    st_o = oracle.store(Lo, C, pool_h, inp.tables_src, jobs, arena_o)
    assert st_o == lmc.LMC_ST_NO_SNAPSHOT
    assert int(st.item()) == st_o
    assert np.array_equal(arena.cpu().numpy(), arena_o)


def test_error_paths_match_oracle(lmc):
    """Bad block ids and bad jobs: same status bits and same arena bytes as
    the oracle (the offending page or object is skipped)."""
    inp, Lp = case_inputs(W.CONFIGS[0])
    Lo, C = inp.layout, inp.C
    pool_h = W.fill_normal_np(Lo.pool_bytes, 3)
    pool = torch.from_numpy(pool_h).to(DEV)
    kda_g = Lo.kv_group_kind.index("KDA")
    mla_g = Lo.kv_group_kind.index("MLA")
    m = C // Lo.N
    cases = []
    for what in ("oor", "neg", "snap", "mla", "req", "align", "end", "chunk", "negchunk", "negoff", "cols"):
        tabs = [t.copy() for t in inp.tables_src]
        jobs = [j.copy() for j in inp.jobs]
        if what == "oor":
            tabs[mla_g][1, 2] = Lo.num_blocks
        elif what == "neg":
            tabs[mla_g][0, 0] = -9
        elif what == "snap":
            tabs[kda_g][1, 2 * m - 1] = -1
        elif what == "mla":
            tabs[mla_g][0, 1] = -1
        elif what == "req":
            jobs[0][1]["request"] = 2
        elif what == "align":
            jobs[1][0]["offset"] += 8
        elif what == "end":
            jobs[1][2]["offset"] = inp.arena_bytes - 16
        elif what == "chunk":
            jobs[0][0]["chunk"] = 1000
        elif what == "negchunk":
            jobs[0][3]["chunk"] = -1
        elif what == "negoff":
            jobs[1][3]["offset"] = -16
        elif what == "cols":
            tabs = [t[:, :3].copy() for t in tabs]
        cases.append((what, tabs, jobs))
    for what, tabs, jobs in cases:
        arena = torch.full((inp.arena_bytes,), 0x77, dtype=torch.uint8, device=DEV)
        st = _status()
        lmc.lmc_store(Lp, C, pool, dev_tables(tabs, DEV), dev_jobs(jobs, DEV), arena, st)
        torch.cuda.synchronize()
        arena_o = np.full(inp.arena_bytes, 0x77, dtype=np.uint8)
        st_o = oracle.store(Lo, C, pool_h, tabs, jobs, arena_o)
        assert st_o != 0, what
        assert int(st.item()) == st_o, (what, int(st.item()), st_o)
        assert np.array_equal(arena.cpu().numpy(), arena_o), what
        # the same faults on the load side
        fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
        st = _status()
        src = torch.from_numpy(arena_o).to(DEV)
        lmc.lmc_load(Lp, C, fresh, dev_tables(tabs, DEV), dev_jobs(jobs, DEV), src, st)
        torch.cuda.synchronize()
        fresh_o = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
        assert oracle.load(Lo, C, fresh_o, tabs, jobs, arena_o) == st_o
        assert int(st.item()) == st_o, what
        assert np.array_equal(fresh.cpu().numpy(), fresh_o), what


def test_status_bits_accumulate(lmc):
    """Status bits are OR-ed into the caller's word, never cleared."""
    inp, Lp = case_inputs(W.CONFIGS[0])
    pool = torch.zeros(inp.layout.pool_bytes, dtype=torch.uint8, device=DEV)
    arena = torch.zeros(inp.arena_bytes, dtype=torch.uint8, device=DEV)
    st = torch.full((1,), 0x100, dtype=torch.int32, device=DEV)
    tabs = [t.copy() for t in inp.tables_src]
    tabs[0][0, 1] = -1
    lmc.lmc_store(Lp, inp.C, pool, dev_tables(tabs, DEV), dev_jobs(inp.jobs, DEV), arena, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0x100 | lmc.LMC_ST_NO_SNAPSHOT


def test_empty_batch_launches_nothing(lmc):
    inp, Lp = case_inputs(W.CONFIGS[0])
    pool = torch.zeros(inp.layout.pool_bytes, dtype=torch.uint8, device=DEV)
    arena = torch.zeros(16, dtype=torch.uint8, device=DEV)
    st = _status()
    empty = [torch.zeros(0, dtype=torch.uint8, device=DEV) for _ in inp.jobs]
    lmc.lmc_store(Lp, inp.C, pool, dev_tables(inp.tables_src, DEV), empty, arena, st)
    lmc.lmc_load(Lp, inp.C, pool, dev_tables(inp.tables_src, DEV), empty, arena, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and not pool.any()


def test_object_at_arena_end(lmc):
    """An object that ends exactly at the arena's last byte is moved."""
    inp, Lp = case_inputs(W.CONFIGS[0])
    Lo, C = inp.layout, inp.C
    pool_h = W.fill_normal_np(Lo.pool_bytes, 4)
    size = inp.object_bytes[1]
    job = np.array([(1, 3, 0)], dtype=W.JOB_DTYPE)
    jobs = [np.zeros(0, dtype=W.JOB_DTYPE), job]
    arena = torch.zeros(size, dtype=torch.uint8, device=DEV)
    st = _status()
    lmc.lmc_store(Lp, C, torch.from_numpy(pool_h).to(DEV), dev_tables(inp.tables_src, DEV),
                  dev_jobs(jobs, DEV), arena, st)
    torch.cuda.synchronize()
    arena_o = np.zeros(size, dtype=np.uint8)
    assert oracle.store(Lo, C, pool_h, inp.tables_src, jobs, arena_o) == 0
    assert int(st.item()) == 0 and np.array_equal(arena.cpu().numpy(), arena_o)


def _oracle_calls(Lo, C):
    return (lambda p, t, j, a: oracle.store(Lo, C, p, t, j, a)), (lambda p, t, j, a: oracle.load(Lo, C, p, t, j, a))


def _full_size(lmc, cfg, request_ids=None):
    """Full-size store + load in the benchmark's launch configuration, every
    byte of both directions compared with the oracle."""
    inp, Lp = case_inputs(cfg, request_ids)
    Lo, C = inp.layout, inp.C
    pool = torch.empty(Lo.pool_bytes, dtype=torch.uint8, device=DEV)
    W.fill_normal(pool, cfg.seed)
    arena = torch.full((inp.arena_bytes,), ARENA_FILL, dtype=torch.uint8, device=DEV)
    fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
    st = _status()
    t_src, t_dst = dev_tables(inp.tables_src, DEV), dev_tables(inp.tables_dst, DEV)
    jobs = dev_jobs(inp.jobs, DEV)
    lmc.lmc_store(Lp, C, pool, t_src, jobs, arena, st)
    lmc.lmc_load(Lp, C, fresh, t_dst, jobs, arena, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    store_o, load_o = _oracle_calls(Lo, C)
    assert check_store_streamed(Lo, C, pool, arena, inp.jobs, inp.object_bytes, inp.tables_src,
                                store_o) == inp.payload_bytes
    del pool
    assert check_load_streamed(Lo, C, fresh, arena, inp.jobs, inp.object_bytes, inp.tables_dst,
                               load_o) == inp.payload_bytes
    torch.cuda.empty_cache()
    # store after load, under the load's tables, reproduces every object
    again = torch.full_like(arena, ARENA_FILL)
    lmc.lmc_store(Lp, C, fresh, t_dst, jobs, again, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(arena, again)
    del arena, again
    torch.cuda.empty_cache()
    assert check_untouched(inp, fresh, inp.jobs, inp.tables_dst, inp.arena_bytes, W.SENTINEL)


def test_full_size_kimi_linear_padded(lmc):
    _full_size(lmc, W.CONFIGS[1])


def test_full_size_kimi_linear_packed_lognormal(lmc):
    _full_size(lmc, W.CONFIGS[2])


@pytest.mark.parametrize("wave", range(4))
def test_full_size_k3_waves(lmc, wave):
    """K3 (93 layers, N = 768, chunk 1536), 4 requests of 131,072 tokens in
    4 waves of one request (a wave's pool, objects and fresh pool fill
    ~116 GB)."""
    _full_size(lmc, W.CONFIGS[3], request_ids=[wave])


def _mixed_run(lmc, inp, Lp, pool, load_arena):
    """The mixed serving step: load of cached chunks on one stream, store of
    new chunks on another, both on the same pool (disjoint blocks, checked
    by the library's guard first, as a caller would)."""
    assert lmc.lmc_check_disjoint(Lp, inp.C, inp.tables_src, inp.load_jobs, inp.tables_src, inp.store_jobs) == -1
    store_arena = torch.full((inp.store_arena_bytes,), ARENA_FILL, dtype=torch.uint8, device=DEV)
    st = _status()
    tabs = dev_tables(inp.tables_src, DEV)
    lj, sj = dev_jobs(inp.load_jobs, DEV), dev_jobs(inp.store_jobs, DEV)
    sa, sb = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    fork = torch.cuda.Event()
    fork.record()
    sa.wait_event(fork)
    sb.wait_event(fork)
    lmc.lmc_load(Lp, inp.C, pool, tabs, lj, load_arena, st, sa)
    lmc.lmc_store(Lp, inp.C, pool, tabs, sj, store_arena, st, sb)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return store_arena, tabs, lj


def test_mixed_step_exact_first_requests(lmc):
    """The mixed step on the first 24 requests, compared in full."""
    inp, Lp = case_inputs(W.CONFIGS[4], request_ids=list(range(24)))
    Lo, C = inp.layout, inp.C
    pool_h = W.fill_normal_np(Lo.pool_bytes, 41)
    load_h = W.fill_normal_np(inp.load_arena_bytes, 42)
    pool = torch.from_numpy(pool_h).to(DEV)
    store_arena, _, _ = _mixed_run(lmc, inp, Lp, pool, torch.from_numpy(load_h).to(DEV))
    # the oracle, in either order: the blocks are disjoint
    assert oracle.load(Lo, C, pool_h, inp.tables_src, inp.load_jobs, load_h) == 0
    store_o = np.zeros(inp.store_arena_bytes, dtype=np.uint8)
    assert oracle.store(Lo, C, pool_h, inp.tables_src, inp.store_jobs, store_o) == 0
    assert np.array_equal(pool.cpu().numpy(), pool_h)
    assert np.array_equal(store_arena.cpu().numpy(), store_o)


def test_mixed_step_block_objects_exact(lmc):
    """The mixed step with block-granular objects: the cached chunks' load
    and the new chunks' store as objects of C / N blocks from their first
    block, then the same with one KDA snapshot per block (last-block and
    every-block forms), issued together on two streams after the library's
    block-form guard; compared in full with the oracle."""
    inp, Lp = case_inputs(W.CONFIGS[4], request_ids=list(range(24)))
    Lo, C = inp.layout, inp.C
    m = C // Lo.N
    for every in (False, True):
        mode = lmc.LMC_KDA_EVERY_BLOCK if every else lmc.LMC_KDA_LAST_BLOCK
        sizes = [Lo.object_bytes_blocks(m, every, g) for g in range(Lo.num_object_groups)]
        units = lambda jobs: [[(int(j["request"]), int(j["chunk"]) * m) for j in J] for J in jobs]
        # the load side holds only the hit boundary's KDA snapshot, so its
        # KDA objects keep the last-block form
        lj, ln = W.pack_jobs(units(inp.load_jobs), [Lo.object_bytes_blocks(m, False, g)
                                                    for g in range(Lo.num_object_groups)])
        sj, sn = W.pack_jobs(units(inp.store_jobs), sizes)
        assert lmc.lmc_check_disjoint_blocks(Lp, m, lmc.LMC_KDA_LAST_BLOCK, inp.tables_src, lj,
                                             inp.tables_src, sj) == -1
        assert lmc.lmc_check_disjoint_blocks(Lp, m, mode, inp.tables_src, sj, inp.tables_src, lj) == -1
        pool_h = W.fill_normal_np(Lo.pool_bytes, 43 + every)
        load_h = W.fill_normal_np(ln, 44 + every)
        pool = torch.from_numpy(pool_h).to(DEV)
        load_arena = torch.from_numpy(load_h).to(DEV)
        store_arena = torch.full((sn,), ARENA_FILL, dtype=torch.uint8, device=DEV)
        st = _status()
        tabs = dev_tables(inp.tables_src, DEV)
        # the job arrays stay referenced until the synchronize: the kernels
        # read them on other streams
        d_lj, d_sj = dev_jobs(lj, DEV), dev_jobs(sj, DEV)
        sa, sb = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
        fork = torch.cuda.Event()
        fork.record()
        sa.wait_event(fork)
        sb.wait_event(fork)
        lmc.lmc_load_blocks(Lp, m, lmc.LMC_KDA_LAST_BLOCK, pool, tabs, d_lj, load_arena, st, sa)
        lmc.lmc_store_blocks(Lp, m, mode, pool, tabs, d_sj, store_arena, st, sb)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert oracle.load_blocks(Lo, m, False, pool_h, inp.tables_src, lj, load_h) == 0
        store_o = np.full(sn, ARENA_FILL, dtype=np.uint8)
        assert oracle.store_blocks(Lo, m, every, pool_h, inp.tables_src, sj, store_o) == 0
        assert np.array_equal(pool.cpu().numpy(), pool_h)
        assert np.array_equal(store_arena.cpu().numpy(), store_o)


def test_temporaries_passed_to_side_streams_stay_valid(lmc):
    """Job arrays built inline for calls on side streams are freed by Python
    as soon as the calls return; the binding marks every tensor it hands to
    a non-current stream as used by that stream, so torch's allocator cannot
    give their memory to the next allocation while the kernels still read
    it. The mixed step written that way (load of cached chunks and store of
    new chunks, temporaries everywhere) is exact against the oracle."""
    inp, Lp = case_inputs(W.CONFIGS[4], request_ids=list(range(24)))
    Lo, C = inp.layout, inp.C
    pool_h = W.fill_normal_np(Lo.pool_bytes, 45)
    load_h = W.fill_normal_np(inp.load_arena_bytes, 46)
    pool = torch.from_numpy(pool_h).to(DEV)
    load_arena = torch.from_numpy(load_h).to(DEV)
    store_arena = torch.full((inp.store_arena_bytes,), ARENA_FILL, dtype=torch.uint8, device=DEV)
    st = _status()
    sa, sb = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    for _ in range(3):
        fork = torch.cuda.Event()
        fork.record()
        sa.wait_event(fork)
        sb.wait_event(fork)
        lmc.lmc_load(Lp, C, pool, dev_tables(inp.tables_src, DEV), dev_jobs(inp.load_jobs, DEV), load_arena, st, sa)
        lmc.lmc_store(Lp, C, pool, dev_tables(inp.tables_src, DEV), dev_jobs(inp.store_jobs, DEV), store_arena, st,
                      sb)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert oracle.load(Lo, C, pool_h, inp.tables_src, inp.load_jobs, load_h) == 0
    store_o = np.full(inp.store_arena_bytes, ARENA_FILL, dtype=np.uint8)
    assert oracle.store(Lo, C, pool_h, inp.tables_src, inp.store_jobs, store_o) == 0
    assert np.array_equal(pool.cpu().numpy(), pool_h)
    assert np.array_equal(store_arena.cpu().numpy(), store_o)


def test_full_size_mixed_two_streams(lmc):
    """The full mixed step: 256 requests, 3 object groups (KDA, SWA-4096,
    MLA), load of hits concurrent with the store of new chunks."""
    cfg = W.CONFIGS[4]
    inp, Lp = case_inputs(cfg)
    Lo, C = inp.layout, inp.C
    pool = torch.empty(Lo.pool_bytes, dtype=torch.uint8, device=DEV)
    W.fill_normal(pool, 40)
    load_arena = torch.empty(inp.load_arena_bytes, dtype=torch.uint8, device=DEV)
    W.fill_normal(load_arena, 42)
    store_arena, tabs, lj = _mixed_run(lmc, inp, Lp, pool, load_arena)
    # every stored object against the oracle, from the pool's pages (the
    # store's blocks are not the load's: the untouched check below shows
    # they still hold the original bytes); every loaded page against the
    # oracle's scatter of the cached objects
    sizes = inp.object_bytes
    store_o, load_o = _oracle_calls(Lo, C)
    assert check_store_streamed(Lo, C, pool, store_arena, inp.store_jobs, sizes, inp.tables_src, store_o) == \
        sum(int(sizes[g]) * len(j) for g, j in enumerate(inp.store_jobs))
    assert check_load_streamed(Lo, C, pool, load_arena, inp.load_jobs, sizes, inp.tables_src, load_o) == \
        sum(int(sizes[g]) * len(j) for g, j in enumerate(inp.load_jobs))
    del store_arena
    # storing the loaded chunks back reproduces the loaded objects
    again = torch.empty_like(load_arena)
    st = _status()
    lmc.lmc_store(Lp, C, pool, tabs, lj, again, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(again, load_arena)
    del again, load_arena
    torch.cuda.empty_cache()
    # every pool byte outside the loaded pages is the original pool's
    ref = torch.empty_like(pool)
    W.fill_normal(ref, 40)
    pages, s0 = oracle.list_pages(Lo, C, inp.tables_src, inp.load_jobs, inp.load_arena_bytes)
    assert s0 == 0
    for pg in pages:
        lo, n = int(pg["pool_offset"]), int(pg["bytes"])
        ref[lo:lo + n] = pool[lo:lo + n]
    assert torch.equal(ref, pool)


# ---------------------------------------------------------------------------
# Block-granular objects (tails, every-block snapshots) and in-pool copies
# ---------------------------------------------------------------------------

def _block_units(inp, kind):
    """(blocks per object, every-block flag, units per object group)."""
    L, C = inp.layout, inp.C
    m = C // L.N
    og_n = L.num_object_groups
    if kind == "every":
        u = [(r, c * m) for r, Lr in enumerate(inp.lengths) for c in range(int(Lr) // C)]
        return [(m, True, [u] * og_n)]
    tails = {}
    for r, Lr in enumerate(inp.lengths):
        t = int(Lr) // L.N - (int(Lr) // C) * m
        if t > 0:
            tails.setdefault(t, []).append((r, (int(Lr) // C) * m))
    return [(nb, False, [u] * og_n) for nb, u in sorted(tails.items())]


def _blocks_exact(lmc, inp, Lp, kind, d=0):
    """Block-granular objects (d > 0: with INT8 KDA records of rows of d)
    stored and loaded back, compared in full with the oracle."""
    Lo = inp.layout
    shapes = _block_units(inp, kind)
    assert shapes
    for nb, every, units in shapes:
        if d:
            sizes = [Lo.object_bytes_blocks_q8(nb, every, d, g) for g in range(Lo.num_object_groups)]
            assert [Lp.object_bytes_blocks_q8(nb, every, d, g) for g in range(Lo.num_object_groups)] == sizes
        else:
            sizes = [Lo.object_bytes_blocks(nb, every, g) for g in range(Lo.num_object_groups)]
            assert [Lp.object_bytes_blocks(nb, every, g) for g in range(Lo.num_object_groups)] == sizes
        jobs, nbytes = W.pack_jobs(units, sizes)
        mode = lmc.LMC_KDA_EVERY_BLOCK if every else lmc.LMC_KDA_LAST_BLOCK
        pool_h = W.fill_normal_np(Lo.pool_bytes, 55 + nb)
        pool = torch.from_numpy(pool_h).to(DEV)
        arena = torch.full((nbytes,), 0x3C, dtype=torch.uint8, device=DEV)
        fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
        st = _status()
        dj = dev_jobs(jobs, DEV)
        t_src, t_dst = dev_tables(inp.tables_src, DEV), dev_tables(inp.tables_dst, DEV)
        arena_o = np.full(nbytes, 0x3C, dtype=np.uint8)
        fresh_o = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
        if d:
            lmc.lmc_store_blocks_q8(Lp, nb, mode, d, pool, t_src, dj, arena, st)
            lmc.lmc_load_blocks_q8(Lp, nb, mode, d, fresh, t_dst, dj, arena, st)
            assert oracle.store_blocks_q8(Lo, nb, every, d, pool_h, inp.tables_src, jobs, arena_o) == 0
            assert oracle.load_blocks_q8(Lo, nb, every, d, fresh_o, inp.tables_dst, jobs, arena_o) == 0
        else:
            lmc.lmc_store_blocks(Lp, nb, mode, pool, t_src, dj, arena, st)
            lmc.lmc_load_blocks(Lp, nb, mode, fresh, t_dst, dj, arena, st)
            assert oracle.store_blocks(Lo, nb, every, pool_h, inp.tables_src, jobs, arena_o) == 0
            assert oracle.load_blocks(Lo, nb, every, fresh_o, inp.tables_dst, jobs, arena_o) == 0
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(arena.cpu().numpy(), arena_o), (kind, nb)
        assert np.array_equal(fresh.cpu().numpy(), fresh_o), (kind, nb)


def _tail_cfg(seed, packed):
    # chunk 150 -> 192 = 3 blocks of 64: the requests leave 1 or 2 tail blocks
    cfg0 = W.CONFIGS[0]
    return W.Config(300 + seed, "tails", cfg0.layers, N=64, requested_chunk=150, packed=packed,
                    num_requests=4, lengths="fixed", fixed_lengths=(300, 517, 640, 1000), seed=seed)


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("kind", ["tails", "every"])
def test_block_objects_exact(lmc, packed, kind):
    inp, Lp = case_inputs(_tail_cfg(7, packed))
    _blocks_exact(lmc, inp, Lp, kind)


@pytest.mark.parametrize("t", range(6))
def test_block_objects_random_specs(lmc, t):
    rng = np.random.default_rng(2000 + t)
    cfg = _random_cfg(rng, t)
    cfg = W.Config(cfg.index, cfg.name, cfg.layers, N=cfg.N, requested_chunk=3 * cfg.N, packed=cfg.packed,
                   num_requests=cfg.num_requests, lengths="fixed",
                   fixed_lengths=tuple(int(x) + 4 * cfg.N for x in cfg.fixed_lengths), snapshot="block",
                   seed=cfg.seed)
    inp, Lp = case_inputs(cfg, split=bool(t % 2))
    _blocks_exact(lmc, inp, Lp, "every")
    if _block_units(inp, "tails"):
        _blocks_exact(lmc, inp, Lp, "tails")


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("kind", ["tails", "every"])
def test_q8_block_objects_exact(lmc, packed, kind):
    """Block-granular objects with INT8 KDA records (rows of 64): tails past
    the last whole chunk (the last block's snapshot) and chunks with one
    snapshot per block."""
    inp, Lp = case_inputs(_tail_cfg(8, packed))
    _blocks_exact(lmc, inp, Lp, kind, d=64)


@pytest.mark.parametrize("d,rows", [(4, 2400), (12, 800), (128, 16), (512, 20)])
def test_q8_block_objects_row_lengths_exact(lmc, d, rows):
    """Every-block INT8 records for row lengths of each encoder and decoder
    path, single- and multi-tile states."""
    state = {"kind": "KDA", "token_bytes": 0, "conv_bytes": 48, "rec_bytes": 4 * d * rows, "window": 0}
    spec = [state, W.mla(32), dict(state, conv_bytes=64), W.mla(32)]
    cfg = W.Config(450 + d, "q8b", spec, N=8, requested_chunk=16, packed=bool(d % 8), num_requests=3,
                   lengths="fixed", fixed_lengths=(40, 77, 23), seed=d)
    inp, Lp = case_inputs(cfg)
    _blocks_exact(lmc, inp, Lp, "every", d=d)


@pytest.mark.parametrize("t", range(6))
def test_q8_random_specs_exact(lmc, t):
    """Random hybrid models (full attention, sliding windows, KDA states of
    (heads, d, d) fp32 with d = 8 .. 64 and conv windows of whole 16-byte
    units), random N and lengths, padded and packed: chunk objects and
    every-block objects with INT8 records, exact against the oracle."""
    rng = np.random.default_rng(7000 + t)
    spec = P.random_spec(rng, int(rng.integers(2, 8)))
    spec = [l for l in spec if l["kind"] != "KDA"] or [W.mla(32)]
    d = int(rng.choice([8, 16, 32, 64]))
    for _ in range(int(rng.integers(1, 4))):
        spec.insert(int(rng.integers(0, len(spec) + 1)),
                    W.kda(8 * int(rng.integers(1, 9)), 3, int(rng.choice([1, 2, 4])), d))
    N = int(rng.choice([2, 4, 16]))
    lengths = tuple(int(x) for x in rng.integers(N, 30 * N, size=int(rng.integers(1, 5))))
    cfg = W.Config(480 + t, "q8-random", spec, N=N, requested_chunk=int(rng.integers(N, 4 * N)),
                   packed=bool(t % 2), num_requests=len(lengths), lengths="fixed", fixed_lengths=lengths,
                   snapshot="block", seed=t)
    inp, Lp = case_inputs(cfg, split=bool((t // 2) % 2))
    _q8_exact(lmc, inp, Lp, d, W.fill_normal_np(inp.layout.pool_bytes, 70 + t))
    _blocks_exact(lmc, inp, Lp, "every", d=d)
    if _block_units(inp, "tails"):
        _blocks_exact(lmc, inp, Lp, "tails", d=d)


def test_block_objects_full_size_tails(lmc):
    """The lognormal Kimi-Linear batch's tail objects at full size: for each
    request, the whole blocks past its last whole chunk (one to N - 1 of
    them, last-block snapshot), grouped by block count; every object and
    every loaded page against the oracle."""
    cfg = W.CONFIGS[2]
    inp, Lp = case_inputs(cfg)
    Lo, C = inp.layout, inp.C
    pool = torch.empty(Lo.pool_bytes, dtype=torch.uint8, device=DEV)
    W.fill_normal(pool, 78)
    t_src, t_dst = dev_tables(inp.tables_src, DEV), dev_tables(inp.tables_dst, DEV)
    shapes = _block_units(inp, "tails")
    assert shapes
    for nb, every, units in shapes:
        sizes = [Lo.object_bytes_blocks(nb, every, g) for g in range(Lo.num_object_groups)]
        assert [Lp.object_bytes_blocks(nb, every, g) for g in range(Lo.num_object_groups)] == sizes
        jobs, nbytes = W.pack_jobs(units, sizes)
        arena = torch.full((nbytes,), ARENA_FILL, dtype=torch.uint8, device=DEV)
        fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
        st = _status()
        dj = dev_jobs(jobs, DEV)
        lmc.lmc_store_blocks(Lp, nb, lmc.LMC_KDA_LAST_BLOCK, pool, t_src, dj, arena, st)
        lmc.lmc_load_blocks(Lp, nb, lmc.LMC_KDA_LAST_BLOCK, fresh, t_dst, dj, arena, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        payload = sum(sizes[g] * len(J) for g, J in enumerate(jobs))
        assert check_store_streamed(
            Lo, C, pool, arena, jobs, sizes, inp.tables_src,
            lambda p, t, j, a: oracle.store_blocks(Lo, nb, False, p, t, j, a), nb=nb) == payload
        assert check_load_streamed(
            Lo, C, fresh, arena, jobs, sizes, inp.tables_dst,
            lambda p, t, j, a: oracle.load_blocks(Lo, nb, False, p, t, j, a), nb=nb) == payload
        del arena, fresh
        torch.cuda.empty_cache()


def test_q8_block_objects_full_size_every_block(lmc):
    """The lognormal Kimi-Linear batch (packed, chunk 2N) as block objects of
    2 blocks with every snapshot an INT8 record (d = 128): every record and
    every decoded page against the oracle."""
    cfg = W.CONFIGS[2]
    inp, Lp = case_inputs(cfg)
    Lo, C = inp.layout, inp.C
    m, d = C // Lo.N, W.state_row_elems(cfg)
    units = [[(int(j["request"]), int(j["chunk"]) * m) for j in J] for J in inp.jobs]
    sizes = [Lo.object_bytes_blocks_q8(m, True, d, g) for g in range(Lo.num_object_groups)]
    jobs, nbytes = W.pack_jobs(units, sizes)
    pool = torch.empty(Lo.pool_bytes, dtype=torch.uint8, device=DEV)
    W.fill_normal(pool, 64)
    arena = torch.full((nbytes,), ARENA_FILL, dtype=torch.uint8, device=DEV)
    fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
    st = _status()
    dj = dev_jobs(jobs, DEV)
    lmc.lmc_store_blocks_q8(Lp, m, lmc.LMC_KDA_EVERY_BLOCK, d, pool, dev_tables(inp.tables_src, DEV), dj, arena, st)
    lmc.lmc_load_blocks_q8(Lp, m, lmc.LMC_KDA_EVERY_BLOCK, d, fresh, dev_tables(inp.tables_dst, DEV), dj, arena, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert check_store_streamed(
        Lo, C, pool, arena, jobs, sizes, inp.tables_src,
        lambda p, t, j, a: oracle.store_blocks_q8(Lo, m, True, d, p, t, j, a), nb=m, kda_every=True) == \
        sum(sizes[g] * len(J) for g, J in enumerate(jobs))
    del pool
    assert check_load_streamed(
        Lo, C, fresh, arena, jobs, sizes, inp.tables_dst,
        lambda p, t, j, a: oracle.load_blocks_q8(Lo, m, True, d, p, t, j, a), nb=m, kda_every=True) == \
        sum(Lo.object_bytes_blocks(m, True, g) * len(J) for g, J in enumerate(jobs))


def test_block_objects_full_size_every_block(lmc):
    """Kimi-Linear packed, chunk = 2N, objects with one KDA snapshot per block:
    every object and every loaded page against the oracle."""
    cfg = W.CONFIGS[2]
    inp, Lp = case_inputs(cfg)
    Lo, C = inp.layout, inp.C
    nb, every, units = _block_units(inp, "every")[0]
    sizes = [Lo.object_bytes_blocks(nb, every, g) for g in range(Lo.num_object_groups)]
    jobs, nbytes = W.pack_jobs(units, sizes)
    pool = torch.empty(Lo.pool_bytes, dtype=torch.uint8, device=DEV)
    W.fill_normal(pool, 77)
    arena = torch.full((nbytes,), ARENA_FILL, dtype=torch.uint8, device=DEV)
    fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
    st = _status()
    dj = dev_jobs(jobs, DEV)
    t_src, t_dst = dev_tables(inp.tables_src, DEV), dev_tables(inp.tables_dst, DEV)
    lmc.lmc_store_blocks(Lp, nb, lmc.LMC_KDA_EVERY_BLOCK, pool, t_src, dj, arena, st)
    lmc.lmc_load_blocks(Lp, nb, lmc.LMC_KDA_EVERY_BLOCK, fresh, t_dst, dj, arena, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    payload = sum(sizes[g] * len(J) for g, J in enumerate(jobs))
    assert check_store_streamed(
        Lo, C, pool, arena, jobs, sizes, inp.tables_src,
        lambda p, t, j, a: oracle.store_blocks(Lo, nb, True, p, t, j, a), nb=nb, kda_every=True) == payload
    del pool
    assert check_load_streamed(
        Lo, C, fresh, arena, jobs, sizes, inp.tables_dst,
        lambda p, t, j, a: oracle.load_blocks(Lo, nb, True, p, t, j, a), nb=nb, kda_every=True) == payload


def _random_pairs(L, rng, per_group, free_from):
    """Distinct sources below `free_from`, distinct destinations at or above it."""
    src = rng.permutation(free_from)
    dst = free_from + rng.permutation(L.num_blocks - free_from)
    out, k = [], 0
    for g in range(L.num_kv_groups):
        n = min(per_group, (L.num_blocks - free_from) // L.num_kv_groups)
        out.append(np.array(list(zip(src[k:k + n], dst[k:k + n])), dtype=oracle.PAIR_DTYPE).reshape(-1))
        k += n
    return out


@pytest.mark.parametrize("t", range(8))
def test_copy_blocks_exact(lmc, t):
    rng = np.random.default_rng(3000 + t)
    spec = P.random_spec(rng, int(rng.integers(2, 9)))
    N = int(rng.choice([4, 16, 64]))
    packed = bool(t % 2)
    o = oracle.layout(spec, N, packed, int(rng.integers(2, 8)) << 20)
    p = lmc.lmc_layout_build(spec, N, packed, int(o.pool_bytes))
    assert p.num_blocks == o.num_blocks and p.base == o.base
    pairs = _random_pairs(o, rng, 6, o.num_blocks // 2)
    if t == 7:  # faults: -1 and an id past the pool are skipped with their bits
        pairs[0] = np.concatenate([pairs[0], np.array([(-1, 1), (2, o.num_blocks)], dtype=oracle.PAIR_DTYPE)])
    pool_h = W.fill_normal_np(o.pool_bytes, t)
    pool = torch.from_numpy(pool_h).to(DEV)
    st = _status()
    lmc.lmc_copy_blocks(p, pool, [lmc.pairs_to_device(x, DEV) for x in pairs], pairs, st)
    torch.cuda.synchronize()
    st_o = oracle.copy_blocks(o, pool_h, pairs)
    assert int(st.item()) == st_o
    assert np.array_equal(pool.cpu().numpy(), pool_h)


def test_copy_blocks_racing_pairs_refused_nothing_launched(lmc):
    """A batch whose pairs would race (a destination another pair reads, in
    another KV group) is refused before any launch: the pool and the status
    word stay as they were. Split into two calls, the same copies run and
    match the oracle applying them in that order."""
    o = oracle.layout(W.CONFIGS[0].layers, 64, False, 1 << 24)
    p = lmc.lmc_layout_build(W.CONFIGS[0].layers, 64, False, 1 << 24)
    e0 = np.zeros(0, dtype=oracle.PAIR_DTYPE)
    first = [np.array([(1, 9)], dtype=oracle.PAIR_DTYPE), e0, e0, e0]
    second = [e0, e0, np.array([(9, 12)], dtype=oracle.PAIR_DTYPE), e0]
    racing = [first[0], e0, second[2], e0]
    pool_h = W.fill_normal_np(o.pool_bytes, 19)
    pool = torch.from_numpy(pool_h).to(DEV)
    st = torch.full((1,), 0x40, dtype=torch.int32, device=DEV)
    with pytest.raises(lmc.LmcError) as e:
        lmc.lmc_copy_blocks(p, pool, [lmc.pairs_to_device(x, DEV) for x in racing], racing, st)
    assert e.value.code == lmc.LMC_ERR_OVERLAP
    torch.cuda.synchronize()
    assert int(st.item()) == 0x40 and np.array_equal(pool.cpu().numpy(), pool_h)
    for part in (first, second):
        lmc.lmc_copy_blocks(p, pool, [lmc.pairs_to_device(x, DEV) for x in part], part, st)
        assert oracle.copy_blocks(o, pool_h, part) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0x40 and np.array_equal(pool.cpu().numpy(), pool_h)


def test_copy_blocks_full_size_kda_states(lmc):
    """Copy-on-write of every KDA snapshot of the Kimi-Linear batch (768
    pairs over 3 KDA groups, 10 GB) into spare blocks of a larger pool."""
    cfg = W.CONFIGS[1]
    inp, _ = case_inputs(cfg)
    need = inp.layout.num_blocks
    per_block = inp.layout.pool_bytes // need
    o = oracle.layout(cfg.layers, cfg.N, cfg.packed, 2 * need * per_block)
    p = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, 2 * need * per_block)
    assert p.base == o.base and p.num_blocks == 2 * need
    pairs = []
    nxt = need
    for g, kind in enumerate(o.kv_group_kind):
        src = inp.tables_src[g][inp.tables_src[g] >= 0] if kind == "KDA" else np.zeros(0, np.int32)
        pairs.append(np.array([(int(s), nxt + i) for i, s in enumerate(src)], dtype=oracle.PAIR_DTYPE).reshape(-1))
        nxt += len(src)
    pool = torch.empty(o.pool_bytes, dtype=torch.uint8, device=DEV)
    W.fill_normal(pool, 91)
    before = pool.clone()
    st = _status()
    lmc.lmc_copy_blocks(p, pool, [lmc.pairs_to_device(x, DEV) for x in pairs], pairs, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # every destination page holds its source page; every other byte is unchanged
    ref = before
    for g, P_ in enumerate(pairs):
        layers = [i for i in range(len(o.kinds)) if o.kv_group[i] == g]
        for pr in P_:
            for i in layers:
                s0 = o.base[i] + int(pr["src_block"]) * o.stride[i]
                d0 = o.base[i] + int(pr["dst_block"]) * o.stride[i]
                ref[d0:d0 + o.real_bytes[i]] = before[s0:s0 + o.real_bytes[i]]
    assert torch.equal(ref, pool)
    # every copied page against the oracle, run on host copies of the
    # source pages, a slice of pairs at a time
    host = LazyHost(o.pool_bytes)
    checked = 0
    for g, P_ in enumerate(pairs):
        layers = [i for i in range(len(o.kinds)) if o.kv_group[i] == g]
        for k in range(0, len(P_), 64):
            sel = P_[k:k + 64]
            for pr in sel:
                for i in layers:
                    s0 = o.base[i] + int(pr["src_block"]) * o.stride[i]
                    fetch(pool, s0, s0 + o.real_bytes[i], host.a[s0:s0 + o.real_bytes[i]])
            only = [np.zeros(0, dtype=oracle.PAIR_DTYPE) for _ in pairs]
            only[g] = sel
            assert oracle.copy_blocks(o, host.a, only) == 0
            for pr in sel:
                for i in layers:
                    d0 = o.base[i] + int(pr["dst_block"]) * o.stride[i]
                    assert np.array_equal(fetch(pool, d0, d0 + o.real_bytes[i]), host.a[d0:d0 + o.real_bytes[i]])
                    checked += o.real_bytes[i]
            host.release()
    assert checked == sum(len(P_) * sum(o.real_bytes[i] for i in range(len(o.kinds)) if o.kv_group[i] == g)
                          for g, P_ in enumerate(pairs))


# ---------------------------------------------------------------------------
# INT8 per-channel codec of the KDA recurrent state
# ---------------------------------------------------------------------------

def _q8_exact(lmc, inp, Lp, d, pool_h):
    Lo, C = inp.layout, inp.C
    sizes = [Lo.object_bytes_q8(C, d, g) for g in range(Lo.num_object_groups)]
    for g in range(Lo.num_object_groups):
        assert Lp.object_bytes_q8(C, d, g) == sizes[g]
    units = [[(int(j["request"]), int(j["chunk"])) for j in J] for J in inp.jobs]
    jobs, nbytes = W.pack_jobs(units, sizes)
    pool = torch.from_numpy(pool_h).to(DEV)
    arena = torch.full((nbytes,), 0x3C, dtype=torch.uint8, device=DEV)
    fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
    st = _status()
    dj = dev_jobs(jobs, DEV)
    lmc.lmc_store_q8(Lp, C, d, pool, dev_tables(inp.tables_src, DEV), dj, arena, st)
    lmc.lmc_load_q8(Lp, C, d, fresh, dev_tables(inp.tables_dst, DEV), dj, arena, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    arena_o = np.full(nbytes, 0x3C, dtype=np.uint8)
    assert oracle.store_q8(Lo, C, d, pool_h, inp.tables_src, jobs, arena_o) == 0
    fresh_o = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
    assert oracle.load_q8(Lo, C, d, fresh_o, inp.tables_dst, jobs, arena_o) == 0
    a = arena.cpu().numpy()
    if not np.array_equal(a, arena_o):
        bad = np.flatnonzero(a != arena_o)
        raise AssertionError(f"{bad.size} record bytes differ, first at {bad[:8]}")
    assert np.array_equal(fresh.cpu().numpy(), fresh_o)


def test_q8_tiny_workload_exact(lmc):
    """The tiny workload: (4, 64, 64) fp32 states as 256 rows of 64 values."""
    inp, Lp = case_inputs(W.CONFIGS[0])
    _q8_exact(lmc, inp, Lp, 64, W.fill_normal_np(inp.layout.pool_bytes, 61))


@pytest.mark.parametrize("d", [64, 128, 16, 4])
def test_q8_special_rows_exact(lmc, d):
    """Rows that decide the corner cases: all zero, subnormal (the clamp
    decides), exact ties at half steps, products within a few ulps of a half
    step (the encoder must fall back to the IEEE quotient), huge and tiny
    magnitudes; for the grouped (d = 16, 64, 128) and one-row-per-warp (d = 4)
    encoders and both decoder paths."""
    inp, Lp = case_inputs(W.CONFIGS[0])
    Lo = inp.layout
    pool_h = W.fill_normal_np(Lo.pool_bytes, 62)
    rng = np.random.default_rng(9)
    f = pool_h[: (Lo.pool_bytes // 4) * 4].view(np.float32)
    nrows = 64 * 64 // d  # one (64, 64) head of the tiny workload's state
    half = np.float32(100) / np.float32(127)
    seen = set()  # layers of different groups share pages in this padded pool: edit each page once
    for i in range(len(Lo.kinds)):
        if Lo.kinds[i] != "KDA":
            continue
        for b in range(Lo.num_blocks):
            lo = (Lo.base[i] + b * Lo.stride[i] + 4608) // 4
            if lo in seen:
                continue
            seen.add(lo)
            rows = f[lo:lo + nrows * d].reshape(nrows, d)
            rows[0] = 0
            rows[1] = 0
            rows[1, :3] = np.array([190, -189, 37], dtype=np.float32) * np.float32(2.0 ** -149)
            rows[2] = np.arange(d, dtype=np.float32) - np.float32((d - 1) / 2)
            rows[3] = rows[3] * np.float32(1e30)  # large but finite (non-finite input is out of domain)
            rows[4] = rows[4] * np.float32(1e-35)
            rows[5, :] = np.float32(127)
            rows[5, 1::2] = np.float32(2.5)
            rows[6] = rng.choice([-3.5, -2.5, -0.5, 0.5, 1.5, 2.5], d).astype(np.float32)
            rows[6, 0] = 127
            # scale 1: half steps moved by one ulp either way
            k = rng.integers(-120, 120, d).astype(np.float32) + np.float32(0.5)
            rows[7] = np.nextafter(k, k + rng.choice([-1, 1], d).astype(np.float32))
            rows[7, 0] = 127
            # scale 100/127: (k + 1/2) * scale, whose quotients land within a few ulps of k + 1/2
            rows[8] = (rng.integers(-127, 126, d).astype(np.float32) + np.float32(0.5)) * half
            rows[8, 0] = 100
    _q8_exact(lmc, inp, Lp, d, pool_h)


@pytest.mark.parametrize("d,rows", [(4, 16), (16, 128), (128, 16), (4, 2400), (8, 1100), (12, 800),
                                    (20, 68), (24, 340), (96, 68), (256, 36), (500, 24), (512, 20)])
def test_q8_row_lengths_exact(lmc, d, rows):
    """Row lengths of every encoder and decoder path (grouped: 8 .. 256;
    one row per warp: 4, 12, 20, 24, 96, 500, 512; decoder one scale per
    vector for powers of two >= 16, four otherwise), pages of one tile and of
    several with a shorter last tile (4 x 2400, 8 x 1100, 12 x 800)."""
    state = {"kind": "KDA", "token_bytes": 0, "conv_bytes": 48, "rec_bytes": 4 * d * rows, "window": 0}
    spec = [state, W.mla(32), dict(state, conv_bytes=64), W.mla(32)]
    cfg = W.Config(400 + d, "q8", spec, N=8, requested_chunk=16, packed=bool(d % 8), num_requests=3,
                   lengths="fixed", fixed_lengths=(40, 77, 23), seed=d)
    inp, Lp = case_inputs(cfg)
    _q8_exact(lmc, inp, Lp, d, W.fill_normal_np(inp.layout.pool_bytes, d + rows))


def test_q8_error_paths_match_oracle(lmc):
    """The codec kernels under the same faults as the plain copies (bad block
    ids, a missing snapshot, bad jobs): same status bits, same record bytes
    and same decoded pages as the oracle."""
    inp, Lp = case_inputs(W.CONFIGS[0])
    Lo, C, d = inp.layout, inp.C, 64
    sizes = [Lo.object_bytes_q8(C, d, g) for g in range(Lo.num_object_groups)]
    units = [[(int(j["request"]), int(j["chunk"])) for j in J] for J in inp.jobs]
    jobs0, nbytes = W.pack_jobs(units, sizes)
    pool_h = W.fill_normal_np(Lo.pool_bytes, 5)
    pool = torch.from_numpy(pool_h).to(DEV)
    kda_g = Lo.kv_group_kind.index("KDA")
    mla_g = Lo.kv_group_kind.index("MLA")
    og_kda = Lo.object_group[Lo.kinds.index("KDA")]
    m = C // Lo.N
    for what in ("oor", "snap", "mla", "req", "align", "end", "chunk"):
        tabs = [t.copy() for t in inp.tables_src]
        jobs = [j.copy() for j in jobs0]
        if what == "oor":
            tabs[kda_g][0, m - 1] = Lo.num_blocks + 3
        elif what == "snap":
            tabs[kda_g][1, 2 * m - 1] = -1
        elif what == "mla":
            tabs[mla_g][0, 1] = -1
        elif what == "req":
            jobs[og_kda][1]["request"] = 2
        elif what == "align":
            jobs[og_kda][0]["offset"] += 8
        elif what == "end":
            jobs[og_kda][2]["offset"] = nbytes - 16
        elif what == "chunk":
            jobs[og_kda][0]["chunk"] = 1000
        arena = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device=DEV)
        st = _status()
        lmc.lmc_store_q8(Lp, C, d, pool, dev_tables(tabs, DEV), dev_jobs(jobs, DEV), arena, st)
        torch.cuda.synchronize()
        arena_o = np.full(nbytes, 0x5A, dtype=np.uint8)
        st_o = oracle.store_q8(Lo, C, d, pool_h, tabs, jobs, arena_o)
        assert st_o != 0, what
        assert int(st.item()) == st_o, (what, int(st.item()), st_o)
        assert np.array_equal(arena.cpu().numpy(), arena_o), what
        fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
        st = _status()
        lmc.lmc_load_q8(Lp, C, d, fresh, dev_tables(tabs, DEV), dev_jobs(jobs, DEV),
                        torch.from_numpy(arena_o).to(DEV), st)
        torch.cuda.synchronize()
        fresh_o = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
        assert oracle.load_q8(Lo, C, d, fresh_o, tabs, jobs, arena_o) == st_o
        assert int(st.item()) == st_o, what
        assert np.array_equal(fresh.cpu().numpy(), fresh_o), what


def test_q8_without_state_layers_is_the_plain_store(lmc):
    """A model with no KDA layer (full and sliding-window attention only):
    the INT8 calls have nothing to encode and move exactly the plain
    objects."""
    spec = [W.mla(64), W.swa(64, 16), W.mla(64), W.swa(64, 16)]
    cfg = W.Config(470, "attn-only", spec, N=8, requested_chunk=16, packed=True, num_requests=3,
                   lengths="fixed", fixed_lengths=(40, 77, 23), seed=47)
    inp, Lp = case_inputs(cfg)
    Lo, C = inp.layout, inp.C
    for g in range(Lo.num_object_groups):
        assert Lp.object_bytes_q8(C, 64, g) == Lo.object_bytes(C, g)
    pool_h = W.fill_normal_np(Lo.pool_bytes, 48)
    pool = torch.from_numpy(pool_h).to(DEV)
    arena = torch.full((inp.arena_bytes,), 0x3C, dtype=torch.uint8, device=DEV)
    fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
    st = _status()
    dj = dev_jobs(inp.jobs, DEV)
    lmc.lmc_store_q8(Lp, C, 64, pool, dev_tables(inp.tables_src, DEV), dj, arena, st)
    lmc.lmc_load_q8(Lp, C, 64, fresh, dev_tables(inp.tables_dst, DEV), dj, arena, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    arena_o = np.full(inp.arena_bytes, 0x3C, dtype=np.uint8)
    assert oracle.store(Lo, C, pool_h, inp.tables_src, inp.jobs, arena_o) == 0
    fresh_o = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
    assert oracle.load(Lo, C, fresh_o, inp.tables_dst, inp.jobs, arena_o) == 0
    assert np.array_equal(arena.cpu().numpy(), arena_o)
    assert np.array_equal(fresh.cpu().numpy(), fresh_o)


def _q8_full_size(lmc, cfg, request_ids=None, seed=63):
    """Full-size chunk store + load with INT8 KDA records (rows of d = 128):
    every record and every decoded page against the oracle."""
    inp, Lp = case_inputs(cfg, request_ids)
    Lo, C = inp.layout, inp.C
    d = W.state_row_elems(cfg)
    sizes = [Lo.object_bytes_q8(C, d, g) for g in range(Lo.num_object_groups)]
    assert [Lp.object_bytes_q8(C, d, g) for g in range(Lo.num_object_groups)] == sizes
    units = [[(int(j["request"]), int(j["chunk"])) for j in J] for J in inp.jobs]
    jobs, nbytes = W.pack_jobs(units, sizes)
    pool = torch.empty(Lo.pool_bytes, dtype=torch.uint8, device=DEV)
    W.fill_normal(pool, seed)
    arena = torch.full((nbytes,), ARENA_FILL, dtype=torch.uint8, device=DEV)
    fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
    st = _status()
    dj = dev_jobs(jobs, DEV)
    t_src, t_dst = dev_tables(inp.tables_src, DEV), dev_tables(inp.tables_dst, DEV)
    lmc.lmc_store_q8(Lp, C, d, pool, t_src, dj, arena, st)
    lmc.lmc_load_q8(Lp, C, d, fresh, t_dst, dj, arena, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert check_store_streamed(Lo, C, pool, arena, jobs, sizes, inp.tables_src,
                                lambda p, t, j, a: oracle.store_q8(Lo, C, d, p, t, j, a)) == \
        sum(sizes[g] * len(J) for g, J in enumerate(jobs))
    del pool
    assert check_load_streamed(Lo, C, fresh, arena, jobs, sizes, inp.tables_dst,
                               lambda p, t, j, a: oracle.load_q8(Lo, C, d, p, t, j, a)) == inp.payload_bytes
    del arena
    torch.cuda.empty_cache()
    assert check_untouched(inp, fresh, inp.jobs, inp.tables_dst, inp.arena_bytes, W.SENTINEL)


def test_q8_full_size_kimi_linear(lmc):
    """Kimi-Linear full size (32 x 8192 tokens, 18 KDA layers of 32 heads)."""
    _q8_full_size(lmc, W.CONFIGS[1])


def test_q8_full_size_k3_wave(lmc):
    """Kimi K3 (69 KDA layers of 64 heads, 147,456-byte conv windows, fp8
    MLA), one wave of one 131,072-token request: the workload whose page
    describes the compressed checkpoints."""
    _q8_full_size(lmc, W.CONFIGS[3], request_ids=[0], seed=73)


def test_q8_row_scale_every_float(lmc):
    """The encoder's row scale equals the IEEE quotient amax / 127 (CUDA's
    division) bit for bit for every finite non-negative float, and its inverse
    is within 3e-7 of 1 / scale wherever the encoder multiplies (so a product
    x * inv stays within 127.01 * 3e-7 < 4e-5 of x / scale); a random sample
    also matches numpy's binary32 division."""
    top = 0x7F7FFFFF + 1  # bit patterns of 0 .. FLT_MAX
    step = 1 << 27
    rng = np.random.default_rng(127)
    for lo in range(0, top, step):
        hi = min(top, lo + step)
        amax = torch.arange(lo, hi, dtype=torch.int64, device=DEV).to(torch.int32).view(torch.float32)
        scale, inv, ieee = (torch.empty_like(amax) for _ in range(3))
        lmc.lmc_selftest_row_scale(amax, scale, inv, ieee)
        torch.cuda.synchronize()
        same = scale.view(torch.int32) == ieee.view(torch.int32)
        if not bool(same.all()):
            bad = torch.nonzero(~same)[:4, 0] + lo
            raise AssertionError(f"row scale differs from the IEEE quotient at bit patterns {bad.tolist()}")
        mult = inv != 0
        err = (inv[mult].double() * scale[mult].double() - 1.0).abs().max().item() if bool(mult.any()) else 0.0
        assert err <= 3e-7, (lo, err)
        divide = ~mult & (amax != 0)
        assert bool(((amax[divide] < 2.0 ** -100) | (amax[divide] > 2.0 ** 125)).all())
        pick = torch.from_numpy(rng.integers(0, hi - lo, 4096)).to(DEV)
        a_h, s_h = amax[pick].cpu().numpy(), scale[pick].cpu().numpy()
        assert np.array_equal(s_h.view(np.int32), (a_h / np.float32(127)).astype(np.float32).view(np.int32))


def test_bounded_wait_reports_timeout_and_context_survives(lmc):
    """A bounded wait that runs out (an mbarrier nothing completes) sets
    LMC_ST_TIMEOUT; the context stays usable: a store right after it still
    matches the oracle."""
    st = _status()
    lmc.lmc_selftest_wait(st, 1000)
    torch.cuda.synchronize()
    assert int(st.item()) == lmc.LMC_ST_TIMEOUT
    inp, Lp = case_inputs(W.CONFIGS[0])
    _full_exact(lmc, inp, Lp)


def test_odd_page_sizes_blocks_and_copies_exact(lmc):
    """Odd page sizes (not 16-byte multiples) take the byte-wise kernels:
    block-granular objects (tails, every-block snapshots) and in-pool copies."""
    spec = [W.mla(18), {"kind": "KDA", "token_bytes": 0, "conv_bytes": 6, "rec_bytes": 70001, "window": 0},
            W.swa(7, 32), W.mla(18)]
    cfg = W.Config(210, "odd", spec, N=8, requested_chunk=20, packed=True, num_requests=3,
                   lengths="fixed", fixed_lengths=(50, 97, 33), seed=5)
    inp, Lp = case_inputs(cfg)
    _blocks_exact(lmc, inp, Lp, "every")
    _blocks_exact(lmc, inp, Lp, "tails")
    o = inp.layout
    rng = np.random.default_rng(77)
    pairs = _random_pairs(o, rng, 4, o.num_blocks // 2)
    pool_h = W.fill_normal_np(o.pool_bytes, 78)
    pool = torch.from_numpy(pool_h).to(DEV)
    st = _status()
    lmc.lmc_copy_blocks(Lp, pool, [lmc.pairs_to_device(x, DEV) for x in pairs], pairs, st)
    torch.cuda.synchronize()
    assert int(st.item()) == oracle.copy_blocks(o, pool_h, pairs) == 0
    assert np.array_equal(pool.cpu().numpy(), pool_h)


class _MappedHost:
    """Pinned, mapped host memory viewed through its device address (the
    library takes any device-accessible pointer as the arena)."""

    def __init__(self, nbytes):
        torch.zeros(1, device=DEV)
        path = [l.split()[-1] for l in open("/proc/self/maps") if "libcudart.so" in l][0]
        self.rt = rt = ctypes.CDLL(path)
        rt.cudaHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
        rt.cudaHostGetDevicePointer.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p, ctypes.c_uint]
        rt.cudaFreeHost.argtypes = [ctypes.c_void_p]
        h, d = ctypes.c_void_p(), ctypes.c_void_p()
        assert rt.cudaHostAlloc(ctypes.byref(h), nbytes, 2) == 0  # cudaHostAllocMapped
        assert rt.cudaHostGetDevicePointer(ctypes.byref(d), h, 0) == 0
        self.h, self.d, self.n = h.value, d.value, nbytes
        self.host = np.ctypeslib.as_array((ctypes.c_uint8 * nbytes).from_address(self.h))

    is_cuda = False

    def is_pinned(self):
        return True  # page-locked and mapped: the kernels address it directly

    def data_ptr(self):
        return self.d

    def numel(self):
        return self.n

    def element_size(self):
        return 1

    def free(self):
        self.rt.cudaFreeHost(ctypes.c_void_p(self.h))


@pytest.mark.parametrize("cfg_index,ids", [(0, None), (1, [0, 1])])
def test_host_resident_arena_exact(lmc, cfg_index, ids):
    """The arena may live in mapped pinned host memory (a host cache tier):
    the kernels store into and load from it across the host link, with the
    same bytes as the oracle."""
    inp, Lp = case_inputs(W.CONFIGS[cfg_index], request_ids=ids)
    Lo, C = inp.layout, inp.C
    pool_h = W.fill_normal_np(Lo.pool_bytes, 90 + cfg_index)
    pool = torch.from_numpy(pool_h).to(DEV)
    host = _MappedHost(inp.arena_bytes)
    try:
        host.host[:] = 0x3C
        fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
        st = _status()
        jobs = dev_jobs(inp.jobs, DEV)
        lmc.lmc_store(Lp, C, pool, dev_tables(inp.tables_src, DEV), jobs, host, st)
        lmc.lmc_load(Lp, C, fresh, dev_tables(inp.tables_dst, DEV), jobs, host, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        arena_o = np.full(inp.arena_bytes, 0x3C, dtype=np.uint8)
        assert oracle.store(Lo, C, pool_h, inp.tables_src, inp.jobs, arena_o) == 0
        assert np.array_equal(host.host, arena_o)
        fresh_o = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
        assert oracle.load(Lo, C, fresh_o, inp.tables_dst, inp.jobs, arena_o) == 0
        assert np.array_equal(fresh.cpu().numpy(), fresh_o)
    finally:
        host.free()


def test_store_load_captured_in_cuda_graph(lmc):
    """store + load captured into one CUDA graph and replayed: the replay
    moves the same bytes as the oracle (the entry points enqueue only a
    kernel launch on the given stream; the first call on a device caches its
    SM count, so it is made before capture)."""
    inp, Lp = case_inputs(W.CONFIGS[0])
    Lo, C = inp.layout, inp.C
    pool_h = W.fill_normal_np(Lo.pool_bytes, 95)
    pool = torch.from_numpy(pool_h).to(DEV)
    arena = torch.zeros(inp.arena_bytes, dtype=torch.uint8, device=DEV)
    fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
    st = _status()
    t_src, t_dst = dev_tables(inp.tables_src, DEV), dev_tables(inp.tables_dst, DEV)
    jobs = dev_jobs(inp.jobs, DEV)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside capture
        lmc.lmc_store(Lp, C, pool, t_src, jobs, arena, st, side)
    torch.cuda.synchronize()
    arena.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        lmc.lmc_store(Lp, C, pool, t_src, jobs, arena, st, side)
        lmc.lmc_load(Lp, C, fresh, t_dst, jobs, arena, st, side)
    torch.cuda.synchronize()
    assert not arena.any(), "capture must not execute the kernels"
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    arena_o = np.zeros(inp.arena_bytes, dtype=np.uint8)
    assert oracle.store(Lo, C, pool_h, inp.tables_src, inp.jobs, arena_o) == 0
    fresh_o = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
    assert oracle.load(Lo, C, fresh_o, inp.tables_dst, inp.jobs, arena_o) == 0
    assert np.array_equal(arena.cpu().numpy(), arena_o)
    assert np.array_equal(fresh.cpu().numpy(), fresh_o)


def test_codec_and_block_calls_captured_in_cuda_graph(lmc):
    """The INT8 calls and the block-granular INT8 calls enqueue only kernel
    launches as well: captured into a CUDA graph (torch's default, global
    capture mode) and replayed, they write the oracle's bytes."""
    cfg = _tail_cfg(9, False)
    inp, Lp = case_inputs(cfg)
    Lo, C, d = inp.layout, inp.C, 64
    m = C // Lo.N
    og = range(Lo.num_object_groups)
    chunk_units = [[(int(j["request"]), int(j["chunk"])) for j in J] for J in inp.jobs]
    block_units = [[(r, c * m) for r, c in u] for u in chunk_units]
    sizes_c = [Lo.object_bytes_q8(C, d, g) for g in og]
    sizes_b = [Lo.object_bytes_blocks_q8(m, True, d, g) for g in og]
    jobs_c, n_c = W.pack_jobs(chunk_units, sizes_c)
    jobs_b, n_b = W.pack_jobs(block_units, sizes_b)
    pool_h = W.fill_normal_np(Lo.pool_bytes, 96)
    pool = torch.from_numpy(pool_h).to(DEV)
    arena_c = torch.zeros(n_c, dtype=torch.uint8, device=DEV)
    arena_b = torch.zeros(n_b, dtype=torch.uint8, device=DEV)
    fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
    st = _status()
    t_src, t_dst = dev_tables(inp.tables_src, DEV), dev_tables(inp.tables_dst, DEV)
    jc, jb = dev_jobs(jobs_c, DEV), dev_jobs(jobs_b, DEV)
    every = lmc.LMC_KDA_EVERY_BLOCK
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside capture
        lmc.lmc_store_q8(Lp, C, d, pool, t_src, jc, arena_c, st, side)
    torch.cuda.synchronize()
    arena_c.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        lmc.lmc_store_q8(Lp, C, d, pool, t_src, jc, arena_c, st, side)
        lmc.lmc_store_blocks_q8(Lp, m, every, d, pool, t_src, jb, arena_b, st, side)
        lmc.lmc_load_blocks_q8(Lp, m, every, d, fresh, t_dst, jb, arena_b, st, side)
    torch.cuda.synchronize()
    assert not arena_c.any() and not arena_b.any(), "capture must not execute the kernels"
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ac = np.zeros(n_c, dtype=np.uint8)
    assert oracle.store_q8(Lo, C, d, pool_h, inp.tables_src, jobs_c, ac) == 0
    ab = np.zeros(n_b, dtype=np.uint8)
    assert oracle.store_blocks_q8(Lo, m, True, d, pool_h, inp.tables_src, jobs_b, ab) == 0
    fo = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
    assert oracle.load_blocks_q8(Lo, m, True, d, fo, inp.tables_dst, jobs_b, ab) == 0
    assert np.array_equal(arena_c.cpu().numpy(), ac)
    assert np.array_equal(arena_b.cpu().numpy(), ab)
    assert np.array_equal(fresh.cpu().numpy(), fo)


def test_one_layout_shared_by_threads_and_streams(lmc):
    """A built layout is shared by four host threads, each storing its own
    request on its own stream into its own arena, many times over: every
    arena equals the oracle's objects for that request (the calls keep no
    state between them)."""
    import threading
    cfg = W.CONFIGS[0]
    inp, Lp = case_inputs(cfg)
    Lo, C = inp.layout, inp.C
    pool_h = W.fill_normal_np(Lo.pool_bytes, 97)
    pool = torch.from_numpy(pool_h).to(DEV)
    t_src = dev_tables(inp.tables_src, DEV)
    work = []
    for k in range(4):
        r = k % len(inp.lengths)
        units = [[(r, c) for c in range(int(inp.lengths[r]) // C)] for _ in range(Lo.num_object_groups)]
        jobs, nbytes = W.pack_jobs(units, inp.object_bytes)
        work.append((jobs, nbytes, torch.zeros(nbytes, dtype=torch.uint8, device=DEV), _status(),
                     torch.cuda.Stream(DEV)))
    torch.cuda.synchronize()
    errors = []

    def run(k):
        try:
            jobs, nbytes, arena, st, stream = work[k]
            dj = dev_jobs(jobs, DEV)
            for _ in range(25):
                lmc.lmc_store(Lp, C, pool, t_src, dj, arena, st, stream)
            stream.synchronize()
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for jobs, nbytes, arena, st, _ in work:
        assert int(st.item()) == 0
        arena_o = np.zeros(nbytes, dtype=np.uint8)
        assert oracle.store(Lo, C, pool_h, inp.tables_src, jobs, arena_o) == 0
        assert np.array_equal(arena.cpu().numpy(), arena_o)


def test_repeated_full_size_launches_are_deterministic(lmc):
    """Fifty store + load rounds of the full Kimi-Linear batch, plain and
    INT8: every round leaves the arena and the reloaded pool bit-identical
    to the first round's (no race between tiles, CTAs or launches)."""
    cfg = W.CONFIGS[1]
    inp, Lp = case_inputs(cfg)
    Lo, C = inp.layout, inp.C
    d = W.state_row_elems(cfg)
    pool = torch.empty(Lo.pool_bytes, dtype=torch.uint8, device=DEV)
    W.fill_normal(pool, 98)
    ts, td = dev_tables(inp.tables_src, DEV), dev_tables(inp.tables_dst, DEV)
    units = [[(int(j["request"]), int(j["chunk"])) for j in J] for J in inp.jobs]
    jobs_q, n_q = W.pack_jobs(units, [Lo.object_bytes_q8(C, d, g) for g in range(Lo.num_object_groups)])
    for q8, jobs_np, nbytes in ((False, inp.jobs, inp.arena_bytes), (True, jobs_q, n_q)):
        arena = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        fresh = torch.full((Lo.pool_bytes,), W.SENTINEL, dtype=torch.uint8, device=DEV)
        st = _status()
        dj = dev_jobs(jobs_np, DEV)
        first = None
        for it in range(50):
            if q8:
                lmc.lmc_store_q8(Lp, C, d, pool, ts, dj, arena, st)
                lmc.lmc_load_q8(Lp, C, d, fresh, td, dj, arena, st)
            else:
                lmc.lmc_store(Lp, C, pool, ts, dj, arena, st)
                lmc.lmc_load(Lp, C, fresh, td, dj, arena, st)
            if it == 0:
                first = (arena.clone(), fresh.clone())
            elif it % 7 == 0 or it == 49:
                assert torch.equal(arena, first[0]) and torch.equal(fresh, first[1]), (q8, it)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        del arena, fresh, first
        torch.cuda.empty_cache()


def _max_spec():
    """256 layers: 62 sliding windows x 4 layers, 4 MLA, 4 KDA; one KV group
    per spec gives 64 KV groups and 64 object groups (the library's limits)."""
    spec = [W.mla(48)] * 4 + [{"kind": "KDA", "token_bytes": 0, "conv_bytes": 32, "rec_bytes": 512,
                               "window": 0}] * 4
    for k in range(62):
        spec += [W.swa(16 * (1 + k % 3), 4 * (1 + k))] * 4
    return [dict(l) for l in spec]


def test_maximum_layout_exact(lmc):
    spec = _max_spec()
    cfg = W.Config(500, "max", spec, N=4, requested_chunk=8, packed=True, num_requests=3, lengths="fixed",
                   fixed_lengths=(40, 23, 57), seed=11)
    inp, Lp = case_inputs(cfg, split=False)
    assert Lp.num_layers == 256 and Lp.num_kv_groups == 64 and Lp.num_object_groups == 64
    _full_exact(lmc, inp, Lp)
    _blocks_exact(lmc, inp, Lp, "every")


def test_maximum_kda_layout_q8_exact(lmc):
    """256 KDA layers (the layer limit) through the INT8 codec: every KDA
    layer takes two launch-plan entries (its conv window and its state
    rows), 512 in one launch. Chunk and every-block forms, exact against the
    oracle."""
    kda = {"kind": "KDA", "token_bytes": 0, "conv_bytes": 32, "rec_bytes": 8 * 16 * 4, "window": 0}
    cfg = W.Config(501, "max-kda", [dict(kda) for _ in range(256)], N=4, requested_chunk=8, packed=True,
                   num_requests=3, lengths="fixed", fixed_lengths=(40, 23, 57), seed=12)
    inp, Lp = case_inputs(cfg, split=False)
    assert Lp.num_layers == 256 and Lp.num_object_groups == 1
    _q8_exact(lmc, inp, Lp, 16, W.fill_normal_np(inp.layout.pool_bytes, 12))
    _blocks_exact(lmc, inp, Lp, "every", d=16)

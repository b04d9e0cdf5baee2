"""liblmc on the host (no GPU): exported symbols, layout / negotiation /
budget parity with the oracle, and the store/load argument checks that run
before anything is enqueued."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import oracle_pins as P
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "lmc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lmc_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lmc):
    names = _declared()
    assert {"lmc_layout_build", "lmc_layout_query", "lmc_layout_free", "lmc_negotiate_chunk",
            "lmc_store", "lmc_load", "lmc_strerror"} <= set(names)
    so = ctypes.CDLL(lmc.LIB_PATH)
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, missing


def assert_same_layout(p, o):
    for f in ("num_kv_groups", "num_object_groups", "num_slabs", "page_size", "block_stride",
              "num_blocks", "pool_bytes", "kv_group", "slot", "object_group", "kv_group_kind",
              "kv_group_size", "real_bytes", "page_bytes", "base", "stride", "kinds"):
        assert getattr(p, f) == getattr(o, f), f


@pytest.mark.parametrize("cfg_index", sorted(W.CONFIGS))
@pytest.mark.parametrize("packed", [False, True])
def test_layout_matches_oracle_on_workloads(lmc, cfg_index, packed):
    cfg = W.CONFIGS[cfg_index]
    for mem in (1 << 34, 123_456_789_012):
        for split in (True, False):
            for sep in (True, False):
                p = lmc.lmc_layout_build(cfg.layers, cfg.N, packed, mem, split, sep)
                o = oracle.layout(cfg.layers, cfg.N, packed, mem, split, sep)
                assert_same_layout(p, o)
                for C in (cfg.N, 2 * cfg.N, 7 * cfg.N):
                    for g in range(o.num_object_groups):
                        assert p.object_bytes(C, g) == o.object_bytes(C, g)
                assert p.object_group_kind == [cfg.layers[p.object_group.index(g)]["kind"]
                                               for g in range(p.num_object_groups)]


def test_layout_matches_oracle_random(lmc):
    rng = np.random.default_rng(3)
    for t in range(400):
        spec = P.random_spec(rng, int(rng.integers(1, 40)))
        N = int(rng.integers(1, 3000))
        mem = int(rng.integers(0, 1 << 36))
        packed, split, sep = bool(t & 1), bool(t & 2), bool(t & 4)
        try:
            o = oracle.layout(spec, N, packed, mem, split, sep)
        except oracle.OracleError as e:
            with pytest.raises(lmc.LmcError) as ei:
                lmc.lmc_layout_build(spec, N, packed, mem, split, sep)
            assert ei.value.code == e.code
            continue
        assert_same_layout(lmc.lmc_layout_build(spec, N, packed, mem, split, sep), o)


def test_layout_rejects_bad_specs_like_oracle(lmc):
    bad = [
        ([W.mla(0)], 16), ([W.swa(16, 0)], 16), ([{"kind": "KDA", "conv_bytes": 0, "rec_bytes": 0}], 16),
        ([{"kind": "KDA", "conv_bytes": -16, "rec_bytes": 32}], 16), ([W.mla(1 << 40)], 1 << 30),
        ([W.mla(16)], 0), ([W.mla(16)], -4),
    ]
    for spec, N in bad:
        with pytest.raises(oracle.OracleError) as eo:
            oracle.layout(spec, N, False, 1 << 30)
        with pytest.raises(lmc.LmcError) as ep:
            lmc.lmc_layout_build(spec, N, False, 1 << 30)
        assert eo.value.code == ep.value.code, spec
    with pytest.raises(lmc.LmcError) as ep:
        lmc.lmc_layout_build([W.mla(16)] * 257, 16, False, 1 << 30)
    assert ep.value.code == lmc.LMC_ERR_INVALID_ARG


def test_negotiation_golden_values(lmc):
    """The library itself against the negotiation values of tests/golden
    (the pages' chunk sizes, plus requests of 0 and -1: non-strict rises to
    N, strict refuses with INVALID_ARG)."""
    names = {lmc.LMC_ERR_NOT_MULTIPLE: "ERR_NOT_MULTIPLE", lmc.LMC_ERR_INVALID_ARG: "ERR_INVALID_ARG"}
    n = 0
    for req, N, strict, exp in P._rows("negotiation.txt"):
        try:
            got = str(lmc.lmc_negotiate_chunk(int(req), int(N), bool(int(strict))))
        except lmc.LmcError as e:
            got = names.get(e.code, str(e.code))
        assert got == exp, (req, N, strict, got, exp)
        n += 1
    assert n >= 17


def test_negotiation_and_budget_match_oracle(lmc):
    for N in list(range(1, 50)) + [768, 944, 1888, 12288]:
        for req in list(range(-2, 200)) + [1500, 12287, 12288, 12289, 2**62]:
            for strict in (False, True):
                try:
                    o = oracle.negotiate_chunk(req, N, strict)
                except oracle.OracleError as e:
                    with pytest.raises(lmc.LmcError) as ep:
                        lmc.lmc_negotiate_chunk(req, N, strict)
                    assert ep.value.code == e.code
                    continue
                assert lmc.lmc_negotiate_chunk(req, N, strict) == o
    for N in range(-1, 40):
        for B in range(-1, 120):
            for sep in (False, True):
                assert lmc.lmc_check_step_budget(N, B, sep) == oracle.check_step_budget(N, B, sep)
    for tb in (1, 7, 576, 1152):
        for state in (1, 100, 70_144, 1_085_440, 2_170_880, 4_341_760):
            for align in (1, 8, 16, 64):
                assert lmc.lmc_unified_block_size(tb, state, align) == oracle.unified_block_size(tb, state, align)
    assert lmc.lmc_strerror(lmc.LMC_ERR_NOT_MULTIPLE).startswith("LMC_ERR_NOT_MULTIPLE")


def _raw_call(lmc, fn, L, chunk, nkv=None, nog=None, status_off=0, njobs=0, null_jobs=False):
    """Calls lmc_store/lmc_load through ctypes with dummy host pointers: every
    case here fails (or finishes with nothing to do) before any CUDA call."""
    nkv = L.num_kv_groups if nkv is None else nkv
    nog = L.num_object_groups if nog is None else nog
    buf = (ctypes.c_uint8 * 64)()
    addr = ctypes.addressof(buf)
    tables = (lmc.lmc_block_table * max(nkv, 1))(*[lmc.lmc_block_table(addr, 4, 4) for _ in range(nkv)])
    jobs = (ctypes.c_void_p * max(nog, 1))(*[None if null_jobs else addr for _ in range(nog)])
    counts = (ctypes.c_int64 * max(nog, 1))(*[njobs] * nog)
    b = lmc.lmc_batch(2, nkv, tables, nog, 0, jobs, counts)
    return getattr(lmc._lib, fn)(L.handle, chunk, addr, ctypes.byref(b), addr, 64, addr + status_off, None)


@pytest.mark.parametrize("fn", ["lmc_store", "lmc_load"])
def test_store_load_host_checks(lmc, fn):
    cfg = W.CONFIGS[1]
    L = lmc.lmc_layout_build(cfg.layers, cfg.N, False, 1 << 34)
    assert _raw_call(lmc, fn, L, 1000) == lmc.LMC_ERR_NOT_MULTIPLE
    assert _raw_call(lmc, fn, L, 0) == lmc.LMC_ERR_NOT_MULTIPLE
    assert _raw_call(lmc, fn, L, 944, status_off=2) == lmc.LMC_ERR_ALIGN
    assert _raw_call(lmc, fn, L, 944, nkv=3) == lmc.LMC_ERR_INVALID_ARG
    assert _raw_call(lmc, fn, L, 944, nog=1) == lmc.LMC_ERR_INVALID_ARG
    assert _raw_call(lmc, fn, L, 944, njobs=-1) == lmc.LMC_ERR_INVALID_ARG
    assert _raw_call(lmc, fn, L, 944, njobs=3, null_jobs=True) == lmc.LMC_ERR_INVALID_ARG
    # nothing to move: returns OK without touching the device
    assert _raw_call(lmc, fn, L, 944, njobs=0) == lmc.LMC_OK
    assert _raw_call(lmc, fn, L, 944, njobs=0, null_jobs=True) == lmc.LMC_OK


@pytest.mark.parametrize("cfg_index", [0, 1, 3, 4])
def test_block_object_sizes_match_oracle(lmc, cfg_index):
    cfg = W.CONFIGS[cfg_index]
    for sep in (True, False):
        p = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, 1 << 36, True, sep)
        o = oracle.layout(cfg.layers, cfg.N, cfg.packed, 1 << 36, True, sep)
        for nb in (1, 2, 3, 7):
            for every in (False, True):
                for g in range(o.num_object_groups):
                    assert p.object_bytes_blocks(nb, every, g) == o.object_bytes_blocks(nb, every, g)
        for g in range(o.num_object_groups):
            assert p.object_bytes_blocks(2, False, g) == p.object_bytes(2 * cfg.N, g)
    with pytest.raises(lmc.LmcError):
        lmc.lmc_object_bytes_blocks(p, 0, lmc.LMC_KDA_LAST_BLOCK, 0)
    with pytest.raises(lmc.LmcError):
        lmc.lmc_object_bytes_blocks(p, 2, 7, 0)


@pytest.mark.parametrize("fn", ["lmc_store_blocks", "lmc_load_blocks"])
def test_block_store_load_host_checks(lmc, fn):
    cfg = W.CONFIGS[1]
    L = lmc.lmc_layout_build(cfg.layers, cfg.N, False, 1 << 34)
    buf = (ctypes.c_uint8 * 64)()
    addr = ctypes.addressof(buf)
    tables = (lmc.lmc_block_table * L.num_kv_groups)(*[lmc.lmc_block_table(addr, 4, 4)] * L.num_kv_groups)
    jobs = (ctypes.c_void_p * L.num_object_groups)(*[addr] * L.num_object_groups)
    counts = (ctypes.c_int64 * L.num_object_groups)(*[0] * L.num_object_groups)
    b = lmc.lmc_batch(2, L.num_kv_groups, tables, L.num_object_groups, 0, jobs, counts)
    f = getattr(lmc._lib, fn)
    assert f(L.handle, 0, 0, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_ERR_INVALID_ARG
    assert f(L.handle, 2, 5, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_ERR_INVALID_ARG
    assert f(L.handle, 2, 1, addr, ctypes.byref(b), addr, 64, addr + 1, None) == lmc.LMC_ERR_ALIGN
    assert f(L.handle, 2, 1, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_OK  # nothing to move


def test_copy_blocks_host_checks(lmc):
    cfg = W.CONFIGS[1]
    L = lmc.lmc_layout_build(cfg.layers, cfg.N, False, 1 << 34)
    buf = (ctypes.c_uint8 * 64)()
    addr = ctypes.addressof(buf)
    g = L.num_kv_groups
    pairs = (ctypes.c_void_p * g)(*[None] * g)
    counts = (ctypes.c_int64 * g)(*[0] * g)
    f = lmc._lib.lmc_copy_blocks
    B = lambda n=g: ctypes.byref(lmc.lmc_copy_batch(n, 0, pairs, counts, pairs))
    assert f(L.handle, addr, B(), addr, None) == lmc.LMC_OK
    assert f(L.handle, addr, B(g - 1), addr, None) == lmc.LMC_ERR_INVALID_ARG
    assert f(L.handle, addr, B(), addr + 2, None) == lmc.LMC_ERR_ALIGN
    # the host copy of the pairs is required
    assert f(L.handle, addr, ctypes.byref(lmc.lmc_copy_batch(g, 0, pairs, counts, None)), addr, None) \
        == lmc.LMC_ERR_INVALID_ARG
    counts[1] = 3  # pairs given as NULL with a non-zero count
    assert f(L.handle, addr, B(), addr, None) == lmc.LMC_ERR_INVALID_ARG


def _copy_batch_code(lmc, L, host_pairs):
    """The library's return code for copies given only on the host. The pool
    pointer is NULL, so a batch that passes the overlap rule is refused with
    INVALID_ARG just before the launch: nothing is ever launched."""
    g = L.num_kv_groups
    keep = [np.ascontiguousarray(p, dtype=lmc.PAIR_DTYPE) for p in host_pairs]
    harr = (ctypes.c_void_p * g)(*[p.ctypes.data if p.size else None for p in keep])
    counts = (ctypes.c_int64 * g)(*[p.size for p in keep])
    buf = (ctypes.c_uint8 * 64)()
    addr = (ctypes.addressof(buf) + 15) // 16 * 16
    return lmc._lib.lmc_copy_blocks(L.handle, None, ctypes.byref(lmc.lmc_copy_batch(g, 0, harr, counts, harr)),
                                    addr, None)


def _racing_pairs(rng, L):
    """A random batch of pairs with one planted collision: a destination
    repeated, or a destination that is another pair's source (possibly in
    another KV group)."""
    nb, g = L.num_blocks, L.num_kv_groups
    ids = rng.permutation(nb)
    n = int(rng.integers(2, max(3, min(12, nb // 2))))
    src, dst = ids[:n], ids[n:2 * n]
    pairs = [np.array([(s, d)], dtype=oracle.PAIR_DTYPE) for s, d in zip(src, dst)]
    i, j = rng.choice(n, 2, replace=False)
    if rng.random() < 0.5:
        pairs[j]["dst_block"] = pairs[i]["dst_block"]
    else:
        pairs[j]["dst_block"] = pairs[i]["src_block"]
    groups = [[] for _ in range(g)]
    for p in pairs:
        groups[int(rng.integers(0, g))].append(p)
    return [np.concatenate(x) if x else np.zeros(0, dtype=oracle.PAIR_DTYPE) for x in groups]


def test_copy_blocks_refuse_racing_pairs_like_the_oracle(lmc):
    """Copies of one call run concurrently: a destination named twice, or a
    destination that another pair reads, is refused before launch by the
    library and by the oracle alike, with nothing copied by the oracle."""
    rng = np.random.default_rng(23)
    for t in range(60):
        spec = P.random_spec(rng, int(rng.integers(1, 9)))
        N = int(rng.integers(1, 40))
        packed = bool(t % 2)
        o = oracle.layout(spec, N, packed, int(rng.integers(1, 4)) << 20)
        p = lmc.lmc_layout_build(spec, N, packed, int(o.pool_bytes))
        if o.num_blocks < 4:
            continue
        pairs = _racing_pairs(rng, o)
        pool = np.zeros(o.pool_bytes, dtype=np.uint8)
        with pytest.raises(oracle.OracleError) as e:
            oracle.copy_blocks(o, pool, pairs)
        assert e.value.code == oracle.ERR_OVERLAP
        assert not pool.any()
        assert _copy_batch_code(lmc, p, pairs) == lmc.LMC_ERR_OVERLAP
    # src == dst alone is allowed; a pair writing what a no-op pair reads is not
    o = oracle.layout(W.CONFIGS[0].layers, 64, False, 1 << 22)
    p = lmc.lmc_layout_build(W.CONFIGS[0].layers, 64, False, 1 << 22)
    g = o.num_kv_groups
    same = [np.array([(3, 3)], dtype=oracle.PAIR_DTYPE)] + [np.zeros(0, dtype=oracle.PAIR_DTYPE)] * (g - 1)
    assert oracle.copy_blocks(o, np.zeros(o.pool_bytes, np.uint8), same) == 0
    assert _copy_batch_code(lmc, p, same) == lmc.LMC_ERR_INVALID_ARG  # passed the rule; NULL pool refused
    clash = [np.array([(3, 3), (5, 3)], dtype=oracle.PAIR_DTYPE)] + [np.zeros(0, dtype=oracle.PAIR_DTYPE)] * (g - 1)
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(o, np.zeros(o.pool_bytes, np.uint8), clash)
    assert _copy_batch_code(lmc, p, clash) == lmc.LMC_ERR_OVERLAP
    # ids outside the pool copy nothing and take no part in the rule
    skipped = [np.array([(-1, 7), (7, o.num_blocks), (2, 7)], dtype=oracle.PAIR_DTYPE)] + \
        [np.zeros(0, dtype=oracle.PAIR_DTYPE)] * (g - 1)
    assert oracle.copy_blocks(o, np.zeros(o.pool_bytes, np.uint8), skipped) == \
        oracle.ST_NO_BLOCK | oracle.ST_BLOCK_OOR


def test_check_disjoint_matches_oracle(lmc):
    """The mixed step's guard: the block sets two chunk batches touch, by the
    library and by the oracle, on the mixed workload (disjoint by
    construction) and on batches with planted shared blocks."""
    cfg = W.CONFIGS[4]
    C = lmc.lmc_negotiate_chunk(cfg.requested_chunk, cfg.N)
    import functools
    full = W.make_inputs(cfg, functools.partial(oracle.layout, cfg.layers, cfg.N, cfg.packed), C)
    pf = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, full.layout.pool_bytes)
    Tf = full.tables_src
    # the whole mixed workload (256 requests) is disjoint on both sides
    assert oracle.check_disjoint(full.layout, C, Tf, full.load_jobs, Tf, full.store_jobs) == -1
    assert lmc.lmc_check_disjoint(pf, C, Tf, full.load_jobs, Tf, full.store_jobs) == -1
    inp = W.make_inputs(cfg, functools.partial(oracle.layout, cfg.layers, cfg.N, cfg.packed), C, list(range(40)))
    o = inp.layout
    p = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, o.pool_bytes)
    T = inp.tables_src
    assert oracle.check_disjoint(o, C, T, inp.load_jobs, T, inp.store_jobs) == -1
    assert lmc.lmc_check_disjoint(p, C, T, inp.load_jobs, T, inp.store_jobs) == -1
    # a batch against itself shares its smallest block
    both = oracle.check_disjoint(o, C, T, inp.store_jobs, T, inp.store_jobs)
    assert both >= 0 and lmc.lmc_check_disjoint(p, C, T, inp.store_jobs, T, inp.store_jobs) == both
    rng = np.random.default_rng(31)
    for t in range(30):
        # plant: one load job moved onto a store job's (request, chunk), or a
        # table entry of the load side pointed at a block the store reads
        lj = [j.copy() for j in inp.load_jobs]
        tables = [x.copy() for x in T]
        og = int(rng.integers(0, len(lj)))
        sj = inp.store_jobs[og]
        if len(lj[og]) and len(sj) and rng.random() < 0.5:
            k = int(rng.integers(0, len(lj[og])))
            s = sj[int(rng.integers(0, len(sj)))]
            lj[og][k]["request"], lj[og][k]["chunk"] = s["request"], s["chunk"]
        else:
            k = int(rng.integers(0, len(tables)))
            used = tables[k][tables[k] >= 0]
            r, c = np.argwhere(tables[k] >= 0)[int(rng.integers(0, used.size))]
            tables[k][r, c] = int(rng.integers(0, o.num_blocks))
        a = oracle.check_disjoint(o, C, tables, lj, tables, inp.store_jobs)
        assert lmc.lmc_check_disjoint(p, C, tables, lj, tables, inp.store_jobs) == a, t
    with pytest.raises(lmc.LmcError) as e:
        lmc.lmc_check_disjoint(p, C + 1, T, inp.load_jobs, T, inp.store_jobs)
    assert e.value.code == lmc.LMC_ERR_NOT_MULTIPLE
    # block-granular batches (first block position, nb blocks per object), both KDA modes
    for nb in (1, 2, 3):
        for every in (False, True):
            mode = lmc.LMC_KDA_EVERY_BLOCK if every else lmc.LMC_KDA_LAST_BLOCK
            for t in range(8):
                bj = [J.copy() for J in inp.load_jobs]
                sj = [J.copy() for J in inp.store_jobs]
                for J in bj + sj:
                    J["chunk"] = J["chunk"] * int(C // cfg.N) + int(rng.integers(0, 2))
                a = oracle.check_disjoint(o, C, T, bj, T, sj, nb=nb, kda_every=every)
                assert lmc.lmc_check_disjoint_blocks(p, nb, mode, T, bj, T, sj) == a, (nb, every, t)
    with pytest.raises(lmc.LmcError) as e:
        lmc.lmc_check_disjoint_blocks(p, 0, lmc.LMC_KDA_LAST_BLOCK, T, inp.load_jobs, T, inp.store_jobs)
    assert e.value.code == lmc.LMC_ERR_INVALID_ARG


@pytest.mark.parametrize("cfg_index", [0, 1, 3])
def test_q8_object_sizes_match_oracle(lmc, cfg_index):
    cfg = W.CONFIGS[cfg_index]
    p = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, 1 << 36)
    o = oracle.layout(cfg.layers, cfg.N, cfg.packed, 1 << 36)
    for d in (4, 16, 64, 128, 256, 512, 6, 1024, 0):
        for C in (cfg.N, 2 * cfg.N):
            for g in range(o.num_object_groups):
                want = o.object_bytes_q8(C, d, g)
                if want < 0:
                    with pytest.raises(lmc.LmcError) as e:
                        p.object_bytes_q8(C, d, g)
                    assert e.value.code == lmc.LMC_ERR_INVALID_ARG
                else:
                    assert p.object_bytes_q8(C, d, g) == want


@pytest.mark.parametrize("cfg_index", [0, 1, 2, 3, 4])
def test_q8_block_object_sizes_match_oracle(lmc, cfg_index):
    cfg = W.CONFIGS[cfg_index]
    p = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, 1 << 36)
    o = oracle.layout(cfg.layers, cfg.N, cfg.packed, 1 << 36)
    for d in (4, 64, 128, 6, 1024):
        for nb in (1, 2, 7):
            for every in (False, True):
                for g in range(o.num_object_groups):
                    want = o.object_bytes_blocks_q8(nb, every, d, g)
                    if want < 0:
                        with pytest.raises(lmc.LmcError) as e:
                            p.object_bytes_blocks_q8(nb, every, d, g)
                        assert e.value.code == lmc.LMC_ERR_INVALID_ARG
                    else:
                        assert p.object_bytes_blocks_q8(nb, every, d, g) == want, (d, nb, every, g)
    # nb = C / N with the last block's snapshot is the chunk form's object
    if o.object_bytes_q8(cfg.N, 128, 0) > 0:
        for g in range(o.num_object_groups):
            assert p.object_bytes_blocks_q8(1, False, 128, g) == p.object_bytes_q8(cfg.N, 128, g)


def test_q8_blocks_host_checks(lmc):
    cfg = W.CONFIGS[1]
    L = lmc.lmc_layout_build(cfg.layers, cfg.N, False, 1 << 34)
    buf = (ctypes.c_uint8 * 256)()
    addr = (ctypes.addressof(buf) + 15) // 16 * 16
    tables = (lmc.lmc_block_table * L.num_kv_groups)(*[lmc.lmc_block_table(addr, 4, 4)] * L.num_kv_groups)
    jobs = (ctypes.c_void_p * L.num_object_groups)(*[addr] * L.num_object_groups)
    counts = (ctypes.c_int64 * L.num_object_groups)(*[1] * L.num_object_groups)
    b = lmc.lmc_batch(2, L.num_kv_groups, tables, L.num_object_groups, 0, jobs, counts)
    for fn in (lmc._lib.lmc_store_blocks_q8, lmc._lib.lmc_load_blocks_q8):
        assert fn(L.handle, 2, 1, 100, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_ERR_INVALID_ARG
        assert fn(L.handle, 2, 2, 128, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_ERR_INVALID_ARG
        assert fn(L.handle, 0, 1, 128, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_ERR_INVALID_ARG
        assert fn(L.handle, 2, 1, 128, addr, ctypes.byref(b), addr + 4, 64, addr, None) == lmc.LMC_ERR_ALIGN


def test_q8_host_checks(lmc):
    cfg = W.CONFIGS[1]
    L = lmc.lmc_layout_build(cfg.layers, cfg.N, False, 1 << 34)
    buf = (ctypes.c_uint8 * 256)()
    addr = (ctypes.addressof(buf) + 15) // 16 * 16
    tables = (lmc.lmc_block_table * L.num_kv_groups)(*[lmc.lmc_block_table(addr, 4, 4)] * L.num_kv_groups)
    jobs = (ctypes.c_void_p * L.num_object_groups)(*[addr] * L.num_object_groups)
    counts = (ctypes.c_int64 * L.num_object_groups)(*[1] * L.num_object_groups)
    b = lmc.lmc_batch(2, L.num_kv_groups, tables, L.num_object_groups, 0, jobs, counts)
    for fn in (lmc._lib.lmc_store_q8, lmc._lib.lmc_load_q8):
        assert fn(L.handle, 944, 100, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_ERR_INVALID_ARG
        assert fn(L.handle, 944, 1024, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_ERR_INVALID_ARG
        assert fn(L.handle, 900, 128, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_ERR_NOT_MULTIPLE
        # the codec moves 16-byte vectors: an unaligned arena is refused before launch
        assert fn(L.handle, 944, 128, addr, ctypes.byref(b), addr + 4, 64, addr, None) == lmc.LMC_ERR_ALIGN


def test_backend_rule_matches_oracle(lmc):
    rng = np.random.default_rng(17)
    cases = [(W.CONFIGS[i].layers, W.CONFIGS[i].N) for i in range(5)]
    cases += [(P.random_spec(rng, int(rng.integers(1, 12))), int(rng.integers(1, 200))) for _ in range(60)]
    for spec, N in cases:
        for packed in (False, True):
            o = oracle.layout(spec, N, packed, 1 << 40)
            p = lmc.lmc_layout_build(spec, N, packed, 1 << 40)
            for a in (False, True):
                for b in (False, True):
                    assert p.check_backends(a, b) == o.check_backends(a, b), (spec, N, packed, a, b)


def test_selftest_wait_host_checks(lmc):
    buf = (ctypes.c_uint8 * 16)()
    addr = ctypes.addressof(buf)
    assert lmc._lib.lmc_selftest_wait(addr, 0, None) == lmc.LMC_ERR_INVALID_ARG
    assert lmc._lib.lmc_selftest_wait(addr, 1 << 30, None) == lmc.LMC_ERR_INVALID_ARG
    assert lmc._lib.lmc_selftest_wait(None, 10, None) == lmc.LMC_ERR_INVALID_ARG
    assert lmc._lib.lmc_selftest_wait((addr + 3) // 4 * 4 + 1, 10, None) == lmc.LMC_ERR_ALIGN


def test_selftest_row_scale_host_checks(lmc):
    buf = (ctypes.c_uint8 * 64)()
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    f = lmc._lib.lmc_selftest_row_scale
    assert f(a, a + 16, a + 32, a + 48, -1, None) == lmc.LMC_ERR_INVALID_ARG
    assert f(None, a + 16, a + 32, a + 48, 4, None) == lmc.LMC_ERR_INVALID_ARG
    assert f(a, a + 16, None, a + 48, 4, None) == lmc.LMC_ERR_INVALID_ARG
    assert f(a + 2, a + 16, a + 32, a + 48, 4, None) == lmc.LMC_ERR_ALIGN
    assert f(a, a + 16, a + 32, a + 48, 0, None) == lmc.LMC_OK  # nothing to do: no launch


def test_q8_refuses_unaligned_state_pages(lmc):
    """A KDA layer without a conv window whose pages sit at odd offsets (an
    odd-sized attention page pads the padded layout) cannot go through the
    16-byte codec: the call is refused before launch."""
    spec = [{"kind": "KDA", "token_bytes": 0, "conv_bytes": 0, "rec_bytes": 4096, "window": 0}, W.mla(17)]
    L = lmc.lmc_layout_build(spec, 300, False, 1 << 24)  # page = 5100 bytes: not a 16-byte multiple
    assert L.page_size % 16 != 0
    buf = (ctypes.c_uint8 * 256)()
    addr = (ctypes.addressof(buf) + 15) // 16 * 16
    tables = (lmc.lmc_block_table * L.num_kv_groups)(*[lmc.lmc_block_table(addr, 4, 4)] * L.num_kv_groups)
    jobs = (ctypes.c_void_p * L.num_object_groups)(*[addr] * L.num_object_groups)
    counts = (ctypes.c_int64 * L.num_object_groups)(*[0] * L.num_object_groups)
    counts[L.object_group[0]] = 1  # only the KDA group has a job
    b = lmc.lmc_batch(1, L.num_kv_groups, tables, L.num_object_groups, 0, jobs, counts)
    assert lmc._lib.lmc_store_q8(L.handle, 300, 16, addr, ctypes.byref(b), addr, 4096, addr, None) \
        == lmc.LMC_ERR_ALIGN


def test_store_refuses_layouts_past_the_launch_limits(lmc):
    """store/load accept at most 64 KV groups and 64 object groups."""
    spec = [W.mla(16)] + [W.swa(16, 4 * (1 + k)) for k in range(64)]  # 65 windows classes
    L = lmc.lmc_layout_build(spec, 4, True, 1 << 30, False)
    assert L.num_object_groups == 65 and L.num_kv_groups == 65
    buf = (ctypes.c_uint8 * 64)()
    addr = ctypes.addressof(buf)
    g, o = L.num_kv_groups, L.num_object_groups
    tables = (lmc.lmc_block_table * g)(*[lmc.lmc_block_table(addr, 4, 4)] * g)
    jobs = (ctypes.c_void_p * o)(*[addr] * o)
    counts = (ctypes.c_int64 * o)(*[0] * o)
    b = lmc.lmc_batch(1, g, tables, o, 0, jobs, counts)
    assert lmc._lib.lmc_store(L.handle, 4, addr, ctypes.byref(b), addr, 64, addr, None) == lmc.LMC_ERR_INVALID_ARG


def test_binding_refuses_memory_the_kernels_cannot_address(lmc):
    """Pageable host tensors are refused with INVALID_ARG before any launch:
    the kernels address device memory or pinned host memory only."""
    import torch
    cfg = W.CONFIGS[0]
    C = lmc.lmc_negotiate_chunk(cfg.requested_chunk, cfg.N)
    L = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, 1 << 24)
    pool = torch.zeros(L.pool_bytes, dtype=torch.uint8)
    arena = torch.zeros(1024, dtype=torch.uint8)
    status = torch.zeros(1, dtype=torch.int32)
    tables = [torch.zeros((1, 8), dtype=torch.int32) for _ in range(L.num_kv_groups)]
    jobs = [torch.zeros(0, dtype=torch.uint8) for _ in range(L.num_object_groups)]
    for call in (lambda: lmc.lmc_store(L, C, pool, tables, jobs, arena, status),
                 lambda: lmc.lmc_load(L, C, pool, tables, jobs, arena, status),
                 lambda: lmc.lmc_store_q8(L, C, 64, pool, tables, jobs, arena, status),
                 lambda: lmc.lmc_copy_blocks(L, pool, [torch.zeros(0, dtype=torch.uint8)] * L.num_kv_groups,
                                             [np.zeros(0, dtype=lmc.PAIR_DTYPE)] * L.num_kv_groups, status)):
        with pytest.raises(lmc.LmcError, match="CUDA tensor or pinned host memory") as e:
            call()
        assert e.value.code == lmc.LMC_ERR_INVALID_ARG


def test_layout_too_small_for_one_block(lmc):
    """Memory below one whole block of the layout: NO_MEMORY from the library
    and the oracle alike (padded: S slabs of one page; packed: one stride)."""
    cfg = W.CONFIGS[1]
    for packed in (False, True):
        big = oracle.layout(cfg.layers, cfg.N, packed, 1 << 40)
        one = big.pool_bytes // big.num_blocks
        for mem in (0, 1, one - 1):
            with pytest.raises(lmc.LmcError) as e:
                lmc.lmc_layout_build(cfg.layers, cfg.N, packed, mem)
            assert e.value.code == lmc.LMC_ERR_NO_MEMORY
            with pytest.raises(oracle.OracleError) as o:
                oracle.layout(cfg.layers, cfg.N, packed, mem)
            assert o.value.code == oracle.ERR_NO_MEMORY
        assert lmc.lmc_layout_build(cfg.layers, cfg.N, packed, one).num_blocks == 1


def test_every_declaration_is_documented():
    """Each entry point of include/lmc.h comes with its comment block (the
    passage it follows, arguments, layout, ownership, errors), alone or
    shared with the declarations of its pair (store/load)."""
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lmc.h")).read()
    names = []
    for m in re.finditer(r"LMC_API [^;]*?\b(lmc_\w+)\s*\(", src):
        before = src[:m.start()].rstrip()
        assert before.endswith("*/") or re.search(r"LMC_API[^;]*;\s*$", before), m.group(1)
        names.append(m.group(1))
    assert len(names) >= 20


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except ImportError:
        return True


@pytest.mark.skipif(not _no_gpu(), reason="passes dummy host pointers to launch-capable calls")
def test_store_size_limits_refused_before_launch(lmc):
    """Sizes the launch plan cannot hold are refused on the host: a page of
    2 GiB or more (INVALID_ARG), an object of more than 2^31 tiles, a chunk of
    more than 2^31 blocks (OVERFLOW). Without a GPU, a call that passed the
    checks would fail only at the launch, with LMC_ERR_CUDA."""
    buf = (ctypes.c_uint8 * 256)()
    addr = (ctypes.addressof(buf) + 15) // 16 * 16

    def batch(L):
        tables = (lmc.lmc_block_table * L.num_kv_groups)(*[lmc.lmc_block_table(addr, 4, 4)] * L.num_kv_groups)
        jobs = (ctypes.c_void_p * L.num_object_groups)(*[addr] * L.num_object_groups)
        counts = (ctypes.c_int64 * L.num_object_groups)(*[1] * L.num_object_groups)
        return lmc.lmc_batch(1, L.num_kv_groups, tables, L.num_object_groups, 0, jobs, counts), (tables, jobs, counts)

    store = lmc._lib.lmc_store
    # a 3 GiB KDA state page
    big = [{"kind": "KDA", "token_bytes": 0, "conv_bytes": 0, "rec_bytes": 3 << 30, "window": 0}]
    L = lmc.lmc_layout_build(big, 16, True, 4 << 30)
    b, keep = batch(L)
    assert store(L.handle, 16, addr, ctypes.byref(b), addr, 1 << 40, addr, None) == lmc.LMC_ERR_INVALID_ARG
    # 2 GiB - 1 MiB attention pages (65,504 tiles each), 40,000 of them per object
    page = (2 << 30) - (1 << 20)
    L = lmc.lmc_layout_build([W.mla(page)], 1, True, 4 << 30)
    b, keep = batch(L)
    assert store(L.handle, 40_000, addr, ctypes.byref(b), addr, 1 << 62, addr, None) == lmc.LMC_ERR_OVERFLOW
    # one block more than 2^31 per chunk
    L = lmc.lmc_layout_build([W.mla(16)], 1, True, 1 << 20)
    b, keep = batch(L)
    assert store(L.handle, (1 << 31) + 1, addr, ctypes.byref(b), addr, 1 << 62, addr, None) == lmc.LMC_ERR_OVERFLOW
    # the largest page the plan holds passes every host check and fails only at the launch
    ok = (2 << 30) - (1 << 16)
    L = lmc.lmc_layout_build([{"kind": "KDA", "token_bytes": 0, "conv_bytes": 0, "rec_bytes": ok, "window": 0}],
                             16, True, 4 << 30)
    b, keep = batch(L)
    assert store(L.handle, 16, addr, ctypes.byref(b), addr, 1 << 40, addr, None) == lmc.LMC_ERR_CUDA


def test_check_disjoint_two_blocks_per_chunk_matches_oracle(lmc):
    """The chunk-form guard with two blocks per chunk (KDA, SWA, MLA layers,
    N = 4, chunk 8), on random planted table entries: library and oracle
    name the same smallest shared block."""
    import functools
    layers = []
    for _ in range(2):
        layers += [{"kind": "KDA", "token_bytes": 0, "conv_bytes": 16, "rec_bytes": 64, "window": 0}] * 3
        layers += [W.swa(16, 12), W.mla(16)]
    cfg = W.Config(601, "mixed-small", layers, N=4, requested_chunk=8, packed=True, num_requests=8,
                   lengths="fixed", fixed_lengths=(40, 23, 57, 31, 64, 17, 12, 48), snapshot="block", seed=7,
                   mixed=True)
    C = oracle.negotiate_chunk(8, 4)
    inp = W.make_inputs(cfg, functools.partial(oracle.layout, layers, 4, True), C)
    o = inp.layout
    p = lmc.lmc_layout_build(layers, 4, True, o.pool_bytes)
    rng = np.random.default_rng(8)
    shared = 0
    for t in range(60):
        tables = [x.copy() for x in inp.tables_src]
        if t:
            k = int(rng.integers(0, len(tables)))
            r, c = np.argwhere(tables[k] >= 0)[int(rng.integers(0, int((tables[k] >= 0).sum())))]
            tables[k][r, c] = int(rng.integers(-1, o.num_blocks + 2))  # -1 and ids past the pool too
        want = oracle.check_disjoint(o, C, tables, inp.load_jobs, tables, inp.store_jobs)
        assert lmc.lmc_check_disjoint(p, C, tables, inp.load_jobs, tables, inp.store_jobs) == want, t
        shared += want >= 0
    assert shared >= 5

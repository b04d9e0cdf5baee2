"""Checks that pin the CPU oracle to facts outside itself.

Each check takes an oracle library handle (the real build, or a mutated copy
in the mutation tests) and raises AssertionError when the oracle disagrees
with the pages' printed values, a closed form, an invariant, or the
independent per-token brute force. Run as a script, it runs every check
against the library path given on the command line and exits non-zero on
the first failure.
"""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import brute  # noqa: E402
import workloads as W  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


# ----------------------------------------------------------------------------
# Negotiation and budget
# ----------------------------------------------------------------------------

def check_negotiation_golden(lib):
    for req, N, strict, exp in _rows("negotiation.txt"):
        try:
            got = oracle.negotiate_chunk(int(req), int(N), bool(int(strict)), _lib=lib)
        except oracle.OracleError as e:
            got = {oracle.ERR_NOT_MULTIPLE: "ERR_NOT_MULTIPLE",
                   oracle.ERR_INVALID_ARG: "ERR_INVALID_ARG"}.get(e.code, e.code)
        assert str(got) == exp, (req, N, strict, got, exp)


def check_negotiation_bruteforce(lib):
    # By search: the least multiple of N not below the request.
    for N in range(1, 41):
        for req in list(range(-3, 300)) + [997, 1000]:
            k = 1
            while k * N < req:
                k += 1
            assert oracle.negotiate_chunk(req, N, False, _lib=lib) == k * N, (req, N)
            if req > 0:
                if req % N == 0:
                    assert oracle.negotiate_chunk(req, N, True, _lib=lib) == req
                else:
                    try:
                        oracle.negotiate_chunk(req, N, True, _lib=lib)
                        raise AssertionError("strict accepted a non-multiple")
                    except oracle.OracleError as e:
                        assert e.code == oracle.ERR_NOT_MULTIPLE


def check_negotiation_edges(lib):
    for N in (0, -5):
        try:
            oracle.negotiate_chunk(100, N, False, _lib=lib)
            raise AssertionError("N <= 0 accepted")
        except oracle.OracleError as e:
            assert e.code == oracle.ERR_INVALID_ARG
    try:
        oracle.negotiate_chunk(2**63 - 5, 10, False, _lib=lib)
        raise AssertionError("overflow not reported")
    except oracle.OracleError as e:
        assert e.code == oracle.ERR_OVERFLOW
    assert oracle.negotiate_chunk(2**62, 2**62, False, _lib=lib) == 2**62


def check_budget(lib):
    for N, B, sep, exp in _rows("step_budget.txt"):
        rc = oracle.check_step_budget(int(N), int(B), bool(int(sep)), _lib=lib)
        assert (rc == 0) == (exp == "OK"), (N, B, sep, rc, exp)
    # Exhaustive on small N: allowed iff N <= B < 2N, or B >= 2N with separation.
    for N in range(1, 30):
        for B in range(1, 100):
            for sep in (0, 1):
                ok = (N <= B < 2 * N) or (B >= 2 * N and sep == 1)
                assert (oracle.check_step_budget(N, B, sep, _lib=lib) == 0) == ok, (N, B, sep)


# ----------------------------------------------------------------------------
# Layout
# ----------------------------------------------------------------------------

def _kimi_linear_state(tp):
    return W.kda(12288 // tp, 3, 32 // tp, 128)


def check_page_formulas(lib):
    """MLA page = N * token_bytes and KDA page = conv + recurrent bytes, pinned
    by the Kimi-Linear block sizes (944 at TP 2, 1888 at TP 1): at the page's
    N the attention page covers the state page, and 16 tokens fewer does not."""
    for tp, N in _rows("block_size.txt"):
        tp, N = int(tp), int(N)
        spec = [_kimi_linear_state(tp), W.mla(1152)]
        for n in (N, N - 16):
            L = oracle.layout(spec, n, False, 1 << 40, _lib=lib)
            kda_page, mla_page = L.real_bytes
            assert kda_page == (12288 // tp) * 3 * 2 + (32 // tp) * 128 * 128 * 4
            assert mla_page == n * 1152
            if n == N:
                assert mla_page >= kda_page
                # padded path A: the smaller (KDA) page is padded to the MLA page
                assert L.page_size == mla_page and L.page_bytes == [mla_page, mla_page]
            else:
                assert mla_page < kda_page


def check_unified_block_size(lib):
    """N = the smallest 16-token multiple whose MLA page covers the KDA state
    page: 944 at TP 2 and 1888 at TP 1 for Kimi-Linear."""
    for tp, N in _rows("block_size.txt"):
        tp, N = int(tp), int(N)
        state = (12288 // tp) * 3 * 2 + (32 // tp) * 128 * 128 * 4
        assert oracle.unified_block_size(1152, state, 16, _lib=lib) == N
    # exhaustive on small sizes: smallest multiple of align covering the state
    for tb in range(1, 12):
        for state in range(1, 200):
            for align in (1, 2, 8, 16):
                n = oracle.unified_block_size(tb, state, align, _lib=lib)
                assert n % align == 0 and n * tb >= state and (n - align) * tb < state


def check_k3_groups(lib):
    rows = {r[0]: r[1:] for r in _rows("k3_groups.txt")}
    L = oracle.layout(W.CONFIGS[3].layers, 768, False, 1 << 50, _lib=lib)
    kda_sizes = [s for s, k in zip(L.kv_group_size, L.kv_group_kind) if k == "KDA"]
    mla_sizes = [s for s, k in zip(L.kv_group_size, L.kv_group_kind) if k == "MLA"]
    assert kda_sizes == [int(x) for x in rows["KDA"]], kda_sizes
    assert mla_sizes == [int(x) for x in rows["MLA"]], mla_sizes
    assert L.num_slabs == int(rows["slabs"][0])
    # each group holds consecutive layers of one kind, in model order
    for g in range(L.num_kv_groups):
        members = [i for i in range(93) if L.kv_group[i] == g]
        assert all(L.kinds[i] == L.kv_group_kind[g] for i in members)
        assert [L.slot[i] for i in members] == list(range(len(members)))


def check_closed_forms(lib):
    """Padded page_size = the largest page; packed block_stride = the largest
    group total; num_blocks = memory // (bytes per block)."""
    layers = W.CONFIGS[1].layers
    mem = 13_754_695_680 + 12345
    kda_page = 73_728 + 2_097_152
    mla_page = 944 * 1152
    P = oracle.layout(layers, 944, False, mem, _lib=lib)
    assert P.kv_group_kind == ["KDA", "KDA", "KDA", "MLA"] and P.kv_group_size == [6, 6, 6, 6]
    assert P.num_slabs == 6 and P.page_size == max(kda_page, mla_page) == kda_page
    assert P.num_blocks == mem // (6 * kda_page) == 1056
    assert P.pool_bytes == 1056 * 6 * kda_page
    assert P.num_object_groups == 2 and P.object_group[:4] == [0, 0, 0, 1]
    for i in range(24):
        assert P.base[i] == P.slot[i] * kda_page * P.num_blocks and P.stride[i] == kda_page
    Q = oracle.layout(layers, 944, True, mem, _lib=lib)
    assert Q.block_stride == max(6 * kda_page, 6 * mla_page) == 13_025_280
    assert Q.num_blocks == mem // 13_025_280
    assert Q.page_size == 0 and Q.page_bytes == Q.real_bytes
    # The MLA group's pages sit back to back from offset 0 of the block.
    mla_layers = [i for i in range(24) if Q.kinds[i] == "MLA"]
    assert [Q.base[i] for i in mla_layers] == [t * mla_page for t in range(6)]
    # object sizes for chunk C = N
    assert P.object_bytes(944, 0) == 18 * kda_page
    assert P.object_bytes(944, 1) == 6 * mla_page
    assert P.object_bytes(1888, 1) == 12 * mla_page and P.object_bytes(1888, 0) == 18 * kda_page
    # tiny case: 64 blocks of one 73,728-byte slab
    T = oracle.layout(W.CONFIGS[0].layers, 64, False, 64 * 73_728, _lib=lib)
    assert T.num_slabs == 1 and T.num_kv_groups == 4 and T.page_size == 73_728 and T.num_blocks == 64
    # one group per spec
    G = oracle.layout(layers, 944, False, mem, split_groups=False, _lib=lib)
    assert G.kv_group_size == [18, 6] and G.num_slabs == 18
    # object-group classes: full attention, KDA, and each sliding window
    spec = [W.kda(64, 3, 2, 16), W.swa(64, 4096), W.mla(64), W.swa(64, 512), W.swa(32, 4096)]
    O = oracle.layout(spec, 16, True, 1 << 30, _lib=lib)
    assert O.object_group == [0, 1, 2, 3, 1] and O.num_object_groups == 4
    O1 = oracle.layout(spec, 16, True, 1 << 30, separate_object_groups=False, _lib=lib)
    assert O1.object_group == [0] * 5 and O1.num_object_groups == 1
    # too little memory for one block
    try:
        oracle.layout(layers, 944, True, 13_025_279, _lib=lib)
        raise AssertionError("a pool without one whole block was accepted")
    except oracle.OracleError as e:
        assert e.code == oracle.ERR_NO_MEMORY


def random_spec(rng, n_layers=None):
    n = n_layers or int(rng.integers(1, 9))
    kinds = rng.choice(["MLA", "KDA", "SWA"], size=n)
    tb = int(rng.choice([16, 32, 48]))
    conv = int(rng.choice([0, 48, 96]))
    rec = int(rng.choice([64, 256, 1024]))
    out = []
    for k in kinds:
        if k == "MLA":
            out.append(W.mla(tb))
        elif k == "SWA":
            out.append(W.swa(tb, int(rng.choice([32, 64]))))
        else:
            out.append(W.kda(conv // 6, 3, 1, int(np.sqrt(rec // 4)) or 4) if conv else
                       {"kind": "KDA", "token_bytes": 0, "conv_bytes": 0, "rec_bytes": rec, "window": 0})
    return out


def check_non_overlap(lib, trials=60):
    """Byte-ownership maps. Pages of different blocks never share a byte;
    inside one block, the pages of one KV group's layers never share a byte
    (layers of different groups do alias at the same block id by design: a
    block belongs to one group at a time, path A's shared tensors and path B's
    per-group offsets both rely on that). Every page lies inside the pool, and
    the brute-force layout agrees."""
    rng = np.random.default_rng(7)
    for t in range(trials):
        spec = random_spec(rng)
        N = int(rng.choice([2, 4, 8]))
        packed = bool(t % 2)
        split = bool((t // 2) % 2)
        mem = int(rng.integers(2000, 40000))
        try:
            L = oracle.layout(spec, N, packed, mem, split_groups=split, _lib=lib)
        except oracle.OracleError as e:
            assert e.code == oracle.ERR_NO_MEMORY
            continue
        B = brute.BruteLayout(spec, N, packed, mem, split)
        assert L.num_blocks == B.num_blocks and L.pool_bytes == B.pool_bytes
        assert [L.kv_group[i] for i in range(len(spec))] == [B.kv_group_of[i] for i in range(len(spec))]
        block_owner = np.full(L.pool_bytes, -1, dtype=np.int64)
        group_owner = {g: np.zeros(L.pool_bytes, dtype=bool) for g in range(L.num_kv_groups)}
        for i in range(len(spec)):
            assert L.base[i] == B.tensor_offset[i] and L.stride[i] == B.layer_stride[i]
            g = L.kv_group[i]
            for b in range(L.num_blocks):
                lo = L.base[i] + b * L.stride[i]
                hi = lo + L.real_bytes[i]
                assert 0 <= lo and hi <= L.pool_bytes, (spec, i, b)
                seen = block_owner[lo:hi]
                assert ((seen == -1) | (seen == b)).all(), ("two blocks share a byte", spec, i, b)
                block_owner[lo:hi] = b
                assert not group_owner[g][lo:hi].any(), ("one group's pages overlap", spec, i, b)
                group_owner[g][lo:hi] = True
        if not packed:
            assert L.page_size == max(L.real_bytes)


# ----------------------------------------------------------------------------
# Store and load
# ----------------------------------------------------------------------------

def tiny_case(lib, cfg_index=0, spec=None, N=None, req_chunk=None, packed=None, lengths=None,
              seed=0, snapshot="block", split=True, separate=True):
    cfg = W.CONFIGS[cfg_index]
    if spec is not None:
        cfg = W.Config(99, "random", spec, N, req_chunk, packed, len(lengths), "fixed",
                       tuple(lengths), snapshot=snapshot, seed=seed)
    C = oracle.negotiate_chunk(cfg.requested_chunk, cfg.N, _lib=lib)
    big = oracle.layout(cfg.layers, cfg.N, cfg.packed, 1 << 40, split_groups=split,
                        separate_object_groups=separate, _lib=lib)
    lengths = W.request_lengths(cfg)
    need = W.count_blocks(cfg, big.kv_group_kind, lengths, cfg.N, C)
    nb = cfg.pool_blocks or need
    per_block = big.pool_bytes // big.num_blocks
    L = oracle.layout(cfg.layers, cfg.N, cfg.packed, nb * per_block, split_groups=split,
                      separate_object_groups=separate, _lib=lib)
    assert L.num_blocks == nb
    sizes = [L.object_bytes(C, g) for g in range(L.num_object_groups)]
    jobs, arena_bytes = W.pack_jobs(W.store_units(lengths, C, L.num_object_groups), sizes)
    t_src = W.block_tables(cfg, L.kv_group_kind, lengths, cfg.N, C, nb, cfg.seed)
    t_dst = W.block_tables(cfg, L.kv_group_kind, lengths, cfg.N, C, nb, cfg.seed + 1000)
    pool = W.fill_normal_np(L.pool_bytes, cfg.seed)
    return dict(cfg=cfg, C=C, L=L, lengths=lengths, jobs=jobs, arena_bytes=arena_bytes,
                t_src=t_src, t_dst=t_dst, pool=pool, sizes=sizes, split=split, separate=separate)


def _addressed(L, C, tables, jobs):
    """Byte mask of every pool byte a store/load of `jobs` touches (pure
    reading of the tables; used for the untouched-bytes invariant)."""
    mask = np.zeros(L.pool_bytes, dtype=bool)
    m = C // L.N
    for og, J in enumerate(jobs):
        for job in J:
            r, c = int(job["request"]), int(job["chunk"])
            for i in range(len(L.kinds)):
                if L.object_group[i] != og:
                    continue
                row = tables[L.kv_group[i]][r]
                pos = [(c + 1) * m - 1] if L.kinds[i] == "KDA" else range(c * m, (c + 1) * m)
                for p in pos:
                    lo = L.base[i] + int(row[p]) * L.stride[i]
                    mask[lo:lo + L.real_bytes[i]] = True
    return mask


def check_store_load(lib, case):
    L, C = case["L"], case["C"]
    pool, jobs = case["pool"], case["jobs"]
    arena = np.zeros(case["arena_bytes"], dtype=np.uint8)
    st = oracle.store(L, C, pool, case["t_src"], jobs, arena)
    assert st == 0, st
    # 1) the per-token brute force builds the same objects
    B = brute.BruteLayout(L_spec(case), L.N, L.packed, L.pool_bytes, case["split"])
    arena_b = np.zeros_like(arena)
    brute.store(B, C, pool, case["t_src"], jobs, arena_b, case["separate"])
    assert np.array_equal(arena, arena_b), "store differs from the per-token brute force"
    # 2) load into a sentinel pool under new tables: addressed bytes restored
    #    by the brute force as well, and every other byte keeps the sentinel
    dst = np.full(L.pool_bytes, W.SENTINEL, dtype=np.uint8)
    assert oracle.load(L, C, dst, case["t_dst"], jobs, arena) == 0
    dst_b = np.full(L.pool_bytes, W.SENTINEL, dtype=np.uint8)
    brute.load(B, C, dst_b, case["t_dst"], jobs, arena, case["separate"])
    assert np.array_equal(dst, dst_b), "load differs from the per-token brute force"
    mask = _addressed(L, C, case["t_dst"], jobs)
    assert (dst[~mask] == W.SENTINEL).all(), "load wrote outside its target pages"
    # 3) re-storing from the loaded pool gives the same objects (identity)
    arena2 = np.zeros_like(arena)
    assert oracle.store(L, C, dst, case["t_dst"], jobs, arena2) == 0
    assert np.array_equal(arena, arena2), "store(load(x)) != x"
    # 4) every object byte came from the source pool: objects are non-trivial
    assert arena.any()
    # 5) the page list names exactly the pages the store reads: a pool that
    #    holds only those pages (zeros elsewhere) stores the same objects,
    #    and the listed pieces tile every object without gaps
    pages, st = oracle.list_pages(L, C, case["t_src"], jobs, case["arena_bytes"])
    assert st == 0
    sparse = np.zeros_like(pool)
    for pg in pages:
        lo = int(pg["pool_offset"])
        sparse[lo:lo + int(pg["bytes"])] = pool[lo:lo + int(pg["bytes"])]
    arena3 = np.zeros_like(arena)
    assert oracle.store(L, C, sparse, case["t_src"], jobs, arena3) == 0
    assert np.array_equal(arena, arena3), "page list misses a page the store reads"
    covered = np.zeros(arena.size, dtype=np.int64)
    for pg in pages:
        o = int(pg["object_offset"])
        covered[o:o + int(pg["bytes"])] += 1
    total = sum(case["sizes"][og] * len(J) for og, J in enumerate(jobs))
    assert int((covered == 1).sum()) == total and covered.max() == 1


def L_spec(case):
    return case["cfg"].layers


def check_errors(lib, case):
    """Bad block ids and bad jobs raise their bits and skip only the page or
    the object concerned."""
    L, C = case["L"], case["C"]
    pool, jobs = case["pool"], case["jobs"]
    good = np.zeros(case["arena_bytes"], dtype=np.uint8)
    oracle.store(L, C, pool, case["t_src"], jobs, good)
    kda_g = L.kv_group_kind.index("KDA")
    mla_g = L.kv_group_kind.index("MLA")
    m = C // L.N
    for what, bit in (("oor", oracle.ST_BLOCK_OOR), ("neg", oracle.ST_BLOCK_OOR),
                      ("snap", oracle.ST_NO_SNAPSHOT), ("mla", oracle.ST_NO_BLOCK)):
        tabs = [t.copy() for t in case["t_src"]]
        if what == "oor":
            tabs[mla_g][0, 0] = L.num_blocks
        elif what == "neg":
            tabs[mla_g][0, 0] = -7
        elif what == "snap":
            tabs[kda_g][0, m - 1] = -1
        else:
            tabs[mla_g][0, 0] = -1
        a = np.full(case["arena_bytes"], 0x5A, dtype=np.uint8)
        st = oracle.store(L, C, pool, tabs, jobs, a)
        assert st == bit, (what, st)
        diff = np.flatnonzero(a != good)
        group = kda_g if what == "snap" else mla_g
        skipped = L.real_bytes[L.kv_group.index(group)]  # one page of that group
        assert (a[diff] == 0x5A).all()
        assert diff.size <= skipped and diff.size > 0, (what, diff.size, skipped)
    # bad jobs: request out of range, misaligned offset, offset past the arena,
    # chunk past the table
    for bad in ("req", "align", "end", "chunk"):
        J = [j.copy() for j in jobs]
        if bad == "req":
            J[0][0]["request"] = len(case["lengths"])
        elif bad == "align":
            J[0][0]["offset"] += 8
        elif bad == "end":
            J[0][0]["offset"] = case["arena_bytes"]
        else:
            J[0][0]["chunk"] = 1 << 20
        a = np.zeros(case["arena_bytes"], dtype=np.uint8)
        assert oracle.store(L, C, pool, case["t_src"], J, a) & oracle.ST_BAD_JOB, bad


def _block_jobs(units, sizes):
    """units[og] = list of (request, first block); packed like chunk jobs."""
    return W.pack_jobs(units, sizes)


def check_block_objects(lib):
    cfg0 = W.CONFIGS[0]
    # chunk 150 -> 192 (3 blocks): requests of 300 and 517 tokens leave 1 and
    # 2 whole tail blocks past their last whole chunk
    _check_block_objects(lib, tiny_case(lib, spec=cfg0.layers, N=64, req_chunk=150, packed=False,
                                        lengths=[300, 517], seed=3))
    rng = np.random.default_rng(13)
    for t in range(4):
        spec = random_spec(rng, int(rng.integers(2, 7)))
        spec[0] = W.mla(int(rng.choice([16, 32])))
        spec[-1] = {"kind": "KDA", "token_bytes": 0, "conv_bytes": 48, "rec_bytes": 256, "window": 0}
        lengths = [int(x) for x in rng.integers(20, 90, size=3)]
        _check_block_objects(lib, tiny_case(lib, spec=spec, N=4, req_chunk=12, packed=bool(t % 2),
                                            lengths=lengths, seed=t, split=bool(t // 2)))


def _check_block_objects(lib, case):
    """Block-granular objects: (1) nb = C/N blocks from chunk * m with the
    last-block snapshot are exactly the chunk objects; (2) tail objects (whole
    blocks past the last whole chunk) and (3) chunk objects with one snapshot
    per block agree with the per-token brute force, and load inverts store."""
    L, C = case["L"], case["C"]
    m = C // L.N
    pool, lengths = case["pool"], case["lengths"]
    B = brute.BruteLayout(L_spec(case), L.N, L.packed, L.pool_bytes, case["split"])
    og_n = L.num_object_groups
    # (1) the chunk form as a special case of the block form
    arena_c = np.zeros(case["arena_bytes"], dtype=np.uint8)
    assert oracle.store(L, C, pool, case["t_src"], case["jobs"], arena_c) == 0
    jb = [j.copy() for j in case["jobs"]]
    for j in jb:
        j["chunk"] = j["chunk"] * m
    arena_b = np.zeros_like(arena_c)
    assert oracle.store_blocks(L, m, False, pool, case["t_src"], jb, arena_b) == 0
    assert np.array_equal(arena_c, arena_b), "block form with nb = C/N differs from the chunk form"
    # (2) tails and (3) every-block snapshots
    tails = {}
    for r, Lr in enumerate(lengths):
        full_blocks = int(Lr) // L.N
        t = full_blocks - (int(Lr) // C) * m
        if t > 0:
            tails.setdefault(t, []).append((r, (int(Lr) // C) * m))
    shapes = [(nb, False, [units] * og_n) for nb, units in tails.items()]
    shapes.append((m, True, [[(r, c * m) for r, Lr in enumerate(lengths) for c in range(int(Lr) // C)]] * og_n))
    for nb, every, units in shapes:
        sizes = [L.object_bytes_blocks(nb, every, g) for g in range(og_n)]
        if every:
            kda_og = [L.object_group[i] for i in range(len(L.kinds)) if L.kinds[i] == "KDA"]
            for g in set(kda_og):
                assert sizes[g] == nb * sum(L.real_bytes[i] for i in range(len(L.kinds))
                                            if L.object_group[i] == g)
        jobs, nbytes = _block_jobs(units, sizes)
        arena = np.zeros(nbytes, dtype=np.uint8)
        assert oracle.store_blocks(L, nb, every, pool, case["t_src"], jobs, arena) == 0
        arena_brute = np.zeros_like(arena)
        brute.store(B, C, pool, case["t_src"], jobs, arena_brute, case["separate"], nb=nb, kda_every=every)
        assert np.array_equal(arena, arena_brute), ("block store differs from the brute force", nb, every)
        dst = np.full(L.pool_bytes, W.SENTINEL, dtype=np.uint8)
        assert oracle.load_blocks(L, nb, every, dst, case["t_dst"], jobs, arena) == 0
        dst_b = np.full(L.pool_bytes, W.SENTINEL, dtype=np.uint8)
        brute.load(B, C, dst_b, case["t_dst"], jobs, arena, case["separate"], nb=nb, kda_every=every)
        assert np.array_equal(dst, dst_b), ("block load differs from the brute force", nb, every)
        again = np.zeros_like(arena)
        assert oracle.store_blocks(L, nb, every, dst, case["t_dst"], jobs, again) == 0
        assert np.array_equal(arena, again)
        pages, st = oracle.list_pages(L, C, case["t_dst"], jobs, nbytes, nb=nb, kda_every=every)
        assert st == 0 and int(pages["bytes"].sum()) == sum(sizes[g] * len(j) for g, j in enumerate(jobs))
    assert len(shapes) >= 2


def check_copy_blocks(lib):
    """In-pool block copies agree with the brute force; the destination pages
    equal the source pages; no other byte changes; bad ids raise bits."""
    rng = np.random.default_rng(21)
    for t in range(10):
        spec = random_spec(rng, int(rng.integers(2, 8)))
        N = int(rng.choice([2, 4, 8]))
        try:
            L = oracle.layout(spec, N, bool(t % 2), int(rng.integers(20000, 60000)), split_groups=bool(t % 3),
                              _lib=lib)
        except oracle.OracleError:
            continue
        if L.num_blocks < 4:
            continue
        pool = W.fill_normal_np(L.pool_bytes, t)
        perm = rng.permutation(L.num_blocks)
        half = L.num_blocks // 2
        pairs = []
        for g in range(L.num_kv_groups):
            k = int(rng.integers(0, half // L.num_kv_groups + 1))
            src = perm[:half][rng.choice(half, k, replace=False)] if k else np.zeros(0, int)
            dst = perm[half:][g * (half // L.num_kv_groups):][:k]
            pairs.append(np.array(list(zip(src, dst)), dtype=oracle.PAIR_DTYPE))
        out = pool.copy()
        assert oracle.copy_blocks(L, out, pairs) == 0
        B = brute.BruteLayout(spec, N, L.packed, L.pool_bytes, bool(t % 3))
        ref = pool.copy()
        brute.copy_blocks(B, ref, pairs)
        assert np.array_equal(out, ref), "copy differs from the brute force"
        changed = np.zeros(L.pool_bytes, dtype=bool)
        for g, P in enumerate(pairs):
            for p in P:
                for i in range(len(spec)):
                    if L.kv_group[i] == g:
                        s0 = L.base[i] + int(p["src_block"]) * L.stride[i]
                        d0 = L.base[i] + int(p["dst_block"]) * L.stride[i]
                        n = L.real_bytes[i]
                        assert np.array_equal(out[d0:d0 + n], pool[s0:s0 + n])
                        changed[d0:d0 + n] = True
        assert np.array_equal(out[~changed], pool[~changed])
    L = oracle.layout(W.CONFIGS[0].layers, 64, False, 64 * 73_728, _lib=lib)
    pool = W.fill_normal_np(L.pool_bytes, 1)
    for bad, bit in (((-1, 3), oracle.ST_NO_BLOCK), ((3, L.num_blocks), oracle.ST_BLOCK_OOR),
                     ((-5, 3), oracle.ST_BLOCK_OOR)):
        pairs = [np.zeros(0, dtype=oracle.PAIR_DTYPE) for _ in range(L.num_kv_groups)]
        pairs[1] = np.array([bad, (7, 8)], dtype=oracle.PAIR_DTYPE)
        out = pool.copy()
        assert oracle.copy_blocks(L, out, pairs) == bit
        ref = pool.copy()
        oracle.copy_blocks(L, ref, [pairs[0], pairs[1][1:], pairs[2], pairs[3]])
        assert np.array_equal(out, ref), "a bad pair must skip only itself"


def _q8_case(lib, rows_x, d):
    """A one-layer KDA layout whose single page holds `rows_x` (fp32) after a
    16-byte conv part; returns (layout, pool, tables, jobs, arena size)."""
    rows_x = np.asarray(rows_x, dtype=np.float32).reshape(-1, d)
    spec = [{"kind": "KDA", "token_bytes": 0, "conv_bytes": 16, "rec_bytes": rows_x.size * 4, "window": 0},
            W.mla(16)]
    L = oracle.layout(spec, 1, True, 1 << 20, _lib=lib)
    pool = np.zeros(L.pool_bytes, dtype=np.uint8)
    b = 3
    lo = L.base[0] + b * L.stride[0]
    pool[lo:lo + 16] = np.arange(16, dtype=np.uint8)
    pool[lo + 16:lo + 16 + rows_x.size * 4] = rows_x.view(np.uint8).reshape(-1)
    kda_g, mla_g = L.kv_group[0], L.kv_group[1]
    tables = [None, None]
    tables[kda_g] = np.array([[b]], dtype=np.int32)
    tables[mla_g] = np.array([[5]], dtype=np.int32)
    size = L.object_bytes_q8(1, d, L.object_group[0])
    jobs = [np.zeros(0, dtype=W.JOB_DTYPE) for _ in range(L.num_object_groups)]
    jobs[L.object_group[0]] = np.array([(0, 0, 0)], dtype=W.JOB_DTYPE)
    return L, pool, tables, jobs, size, rows_x, lo


def check_q8_golden(lib):
    """Worked rows: half-to-even ties, clamping at 127, zero rows, exact
    round trips when the scale is a power of two."""
    lines = [l.split("#")[0].strip() for l in open(os.path.join(GOLDEN, "q8_rows.txt"))]
    lines = [l for l in lines if l]
    xs, qs, ss = [], [], []
    for k in range(0, len(lines), 3):
        xs.append(np.array(lines[k].split(":")[1].split(), dtype=np.float32))
        qs.append(np.array(lines[k + 1].split(":")[1].split(), dtype=np.int8))
        ss.append(np.float32(lines[k + 2].split(":")[1]))
    n = len(xs)
    assert n % 4 == 0  # records keep whole groups of 4 rows
    x, q, sc = np.stack(xs), np.stack(qs), np.array(ss, dtype=np.float32)
    L, pool, tables, jobs, size, rows_x, lo = _q8_case(lib, x, 8)
    assert size == 16 + 4 * n + 8 * n
    arena = np.zeros(size, dtype=np.uint8)
    assert oracle.store_q8(L, 1, 8, pool, tables, jobs, arena) == 0
    assert np.array_equal(arena[:16], np.arange(16, dtype=np.uint8)), "conv part must stay raw"
    assert np.array_equal(arena[16:16 + 4 * n].view(np.float32), sc), arena[16:16 + 4 * n].view(np.float32)
    assert np.array_equal(arena[16 + 4 * n:].view(np.int8).reshape(n, 8), q), arena[16 + 4 * n:].view(np.int8)
    back = np.zeros_like(pool)
    assert oracle.load_q8(L, 1, 8, back, tables, jobs, arena) == 0
    got = back[lo + 16:lo + 16 + 32 * n].view(np.float32).reshape(n, 8)
    assert np.array_equal(got, q.astype(np.float32) * sc[:, None])


def q8_numpy(x, d):
    """Independent float32 restatement of the codec for the pins."""
    x = np.asarray(x, dtype=np.float32).reshape(-1, d)
    amax = np.max(np.abs(x), axis=1)
    scale = (amax / np.float32(127)).astype(np.float32)
    safe = np.where(scale == 0, np.float32(1), scale).astype(np.float32)
    q = np.rint((x / safe[:, None]).astype(np.float32))
    q = np.where(scale[:, None] == 0, 0, np.clip(q, -127, 127)).astype(np.int8)
    return scale, q


def check_q8_random(lib):
    """Random N(0,1) states (plus scaled and sparse rows): the C codec equals
    the numpy restatement bit for bit, and every decoded value lies within
    half a step of its input."""
    rng = np.random.default_rng(31)
    for d in (4, 8, 64, 128, 512):
        rows = 4 * int(rng.integers(1, 10)) - 1  # plus the subnormal row below: a multiple of 4
        x = rng.standard_normal((rows, d)).astype(np.float32)
        x[0] *= np.float32(1e-30)
        x[-1, : d // 2] = 0
        # a subnormal row: its scale (max/127) rounds coarsely, so x/scale can
        # exceed 127.5 and the clamp to [-127, 127] decides the code
        sub = np.zeros(d, dtype=np.float32)
        sub[0] = np.float32(190 * 2.0 ** -149)
        sub[1] = -np.float32(189 * 2.0 ** -149)
        sub[2] = np.float32(37 * 2.0 ** -149)
        x = np.vstack([x, sub[None, :]]).astype(np.float32)
        rows += 1
        if rows > 2:
            x[1] = 0
        L, pool, tables, jobs, size, rows_x, lo = _q8_case(lib, x, d)
        arena = np.zeros(size, dtype=np.uint8)
        assert oracle.store_q8(L, 1, d, pool, tables, jobs, arena) == 0
        scale = arena[16:16 + 4 * rows].view(np.float32)
        codes = arena[16 + 4 * rows:16 + 4 * rows + rows * d].view(np.int8).reshape(rows, d)
        s_np, q_np = q8_numpy(x, d)
        assert np.array_equal(scale, s_np) and np.array_equal(codes, q_np)
        back = np.zeros_like(pool)
        assert oracle.load_q8(L, 1, d, back, tables, jobs, arena) == 0
        y = back[lo + 16:lo + 16 + 4 * rows * d].view(np.float32).reshape(rows, d)
        err = np.abs(y.astype(np.float64) - x.astype(np.float64))
        bound = scale.astype(np.float64)[:, None] * (0.5 + 1e-6) + 1e-45
        assert (err[:-1] <= bound[:-1]).all()
        assert (np.abs(codes) <= 127).all()
        assert codes[-1, 0] == 127 and codes[-1, 1] == -127  # clamped (190 and -189 steps)
    # a d that is not accepted is an argument error
    L, pool, tables, jobs, size, rows_x, lo = _q8_case(lib, np.zeros(96, np.float32), 8)
    for bad in (6, 0, 1024, 16, 32, 36):  # 16, 32: 6 and 3 rows (not 4k); 36: not whole rows
        try:
            oracle.store_q8(L, 1, bad, pool, tables, jobs, np.zeros(4096, np.uint8))
            raise AssertionError(f"row length {bad} accepted")
        except oracle.OracleError as e:
            assert e.code == oracle.ERR_INVALID_ARG


def check_q8_objects(lib):
    """In whole objects the codec touches only KDA pages: paged layers are
    byte-identical to the plain store and objects shrink by the codec's
    ratio; store_q8 then load_q8 restores conv bytes exactly and state
    values within half a step."""
    case = tiny_case(lib, 0)
    L, C = case["L"], case["C"]
    d = 64
    sizes = [L.object_bytes_q8(C, d, g) for g in range(L.num_object_groups)]
    kda_og = L.object_group[0]
    rows = (4 * 64 * 64 * 4) // (4 * d)
    assert sizes[kda_og] == 3 * (4608 + 4 * rows + rows * d)
    jobs, nbytes = W.pack_jobs(W.store_units(case["lengths"], C, L.num_object_groups), sizes)
    arena = np.zeros(nbytes, dtype=np.uint8)
    assert oracle.store_q8(L, C, d, case["pool"], case["t_src"], jobs, arena) == 0
    plain = np.zeros(case["arena_bytes"], dtype=np.uint8)
    oracle.store(L, C, case["pool"], case["t_src"], case["jobs"], plain)
    mla_og = 1 - kda_og
    for a, b in zip(jobs[mla_og], case["jobs"][mla_og]):
        n = sizes[mla_og]
        assert np.array_equal(arena[int(a["offset"]):int(a["offset"]) + n], plain[int(b["offset"]):int(b["offset"]) + n])
    dst = np.zeros(L.pool_bytes, dtype=np.uint8)
    assert oracle.load_q8(L, C, d, dst, case["t_dst"], jobs, arena) == 0
    m = C // L.N
    for r, Lr in enumerate(case["lengths"]):
        for c in range(int(Lr) // C):
            for i in range(3):
                g = L.kv_group[i]
                src = L.base[i] + int(case["t_src"][g][r, (c + 1) * m - 1]) * L.stride[i]
                out = L.base[i] + int(case["t_dst"][g][r, (c + 1) * m - 1]) * L.stride[i]
                assert np.array_equal(dst[out:out + 4608], case["pool"][src:src + 4608])
                x = case["pool"][src + 4608:src + 70144].view(np.float32).reshape(-1, d)
                y = dst[out + 4608:out + 70144].view(np.float32).reshape(-1, d)
                s_np, q_np = q8_numpy(x, d)
                assert np.array_equal(y, q_np.astype(np.float32) * s_np[:, None])


def check_q8_block_objects(lib):
    """Block-granular objects with INT8 records: (1) nb = C/N blocks from
    chunk * m with the last-block snapshot are exactly the chunk-form INT8
    objects; (2) with one snapshot per block, each KDA layer holds nb records
    in block order, each its page's raw conv bytes then the numpy
    restatement's scales and codes, while paged layers equal the plain block
    objects; (3) the load restores conv bytes exactly and states as decoded
    codes at every block position; (4) row lengths outside the rules are
    refused."""
    case = tiny_case(lib, 0)
    L, C = case["L"], case["C"]
    m, d = C // L.N, 64
    og_n = L.num_object_groups
    pool = case["pool"]
    units = [[(int(j["request"]), int(j["chunk"]) * m) for j in J] for J in case["jobs"]]
    # (1)
    sizes_c = [L.object_bytes_q8(C, d, g) for g in range(og_n)]
    jobs_c, nbytes = W.pack_jobs(W.store_units(case["lengths"], C, og_n), sizes_c)
    arena_c = np.zeros(nbytes, dtype=np.uint8)
    assert oracle.store_q8(L, C, d, pool, case["t_src"], jobs_c, arena_c) == 0
    sizes_b = [L.object_bytes_blocks_q8(m, False, d, g) for g in range(og_n)]
    assert sizes_b == sizes_c
    jobs_b, nbytes_b = W.pack_jobs(units, sizes_b)
    arena_b = np.zeros(nbytes_b, dtype=np.uint8)
    assert oracle.store_blocks_q8(L, m, False, d, pool, case["t_src"], jobs_b, arena_b) == 0
    assert np.array_equal(arena_c, arena_b), "block INT8 form with nb = C/N differs from the chunk form"
    # (2)
    sizes = [L.object_bytes_blocks_q8(m, True, d, g) for g in range(og_n)]
    plain_sizes = [L.object_bytes_blocks(m, True, g) for g in range(og_n)]
    kda = [i for i in range(len(L.kinds)) if L.kinds[i] == "KDA"]
    conv, rec = 4608, 4 * 64 * 64 * 4
    rows = rec // (4 * d)
    record = conv + 4 * rows + rows * d
    kda_og = L.object_group[kda[0]]
    assert sizes[kda_og] == m * len(kda) * record
    jobs, nbytes = W.pack_jobs(units, sizes)
    arena = np.zeros(nbytes, dtype=np.uint8)
    assert oracle.store_blocks_q8(L, m, True, d, pool, case["t_src"], jobs, arena) == 0
    plain_jobs, plain_bytes = W.pack_jobs(units, plain_sizes)
    plain = np.zeros(plain_bytes, dtype=np.uint8)
    assert oracle.store_blocks(L, m, True, pool, case["t_src"], plain_jobs, plain) == 0
    for g in range(og_n):
        if g == kda_og:
            continue
        for a, b in zip(jobs[g], plain_jobs[g]):
            n = sizes[g]
            assert np.array_equal(arena[int(a["offset"]):int(a["offset"]) + n], plain[int(b["offset"]):int(b["offset"]) + n])
    for job in jobs[kda_og]:
        r, first, off = int(job["request"]), int(job["chunk"]), int(job["offset"])
        for k, i in enumerate(kda):
            for j in range(m):
                rec_at = off + (k * m + j) * record
                blk = int(case["t_src"][L.kv_group[i]][r, first + j])
                page = L.base[i] + blk * L.stride[i]
                assert np.array_equal(arena[rec_at:rec_at + conv], pool[page:page + conv])
                s_np, q_np = q8_numpy(pool[page + conv:page + conv + rec].view(np.float32), d)
                got_s = arena[rec_at + conv:rec_at + conv + 4 * rows].view(np.float32)
                got_q = arena[rec_at + conv + 4 * rows:rec_at + record].view(np.int8).reshape(rows, d)
                assert np.array_equal(got_s, s_np) and np.array_equal(got_q, q_np), (r, first, i, j)
    # (3)
    dst = np.zeros(L.pool_bytes, dtype=np.uint8)
    assert oracle.load_blocks_q8(L, m, True, d, dst, case["t_dst"], jobs, arena) == 0
    for job in jobs[kda_og]:
        r, first = int(job["request"]), int(job["chunk"])
        for i in kda:
            g = L.kv_group[i]
            for j in range(m):
                src = L.base[i] + int(case["t_src"][g][r, first + j]) * L.stride[i]
                out = L.base[i] + int(case["t_dst"][g][r, first + j]) * L.stride[i]
                assert np.array_equal(dst[out:out + conv], pool[src:src + conv])
                s_np, q_np = q8_numpy(pool[src + conv:src + conv + rec].view(np.float32), d)
                y = dst[out + conv:out + conv + rec].view(np.float32).reshape(-1, d)
                assert np.array_equal(y, q_np.astype(np.float32) * s_np[:, None])
    # (4)
    assert L.object_bytes_blocks_q8(m, True, 6, kda_og) == -1
    assert L.object_bytes_blocks_q8(0, True, d, kda_og) == -1
    try:
        oracle.store_blocks_q8(L, m, True, 6, pool, case["t_src"], jobs, np.zeros(nbytes, np.uint8))
        raise AssertionError("row length 6 accepted")
    except oracle.OracleError as e:
        assert e.code == oracle.ERR_INVALID_ARG


def check_backends(lib):
    """vLLM's eligibility rule ("How vLLM manages the KV cache of hybrid
    models", §3.3): Kimi-Linear at its own N pads the KDA page (always
    allowed); the 24-layer workload (N = 944 with a TP-1 state) pads the MLA
    page, which needs stride-indexing attention; packed needs every backend to
    stride, which KDA kernels that assume contiguous pages cannot; a pure
    attention model packs when its backends stride."""
    tp2 = [_kimi_linear_state(2), W.mla(1152)]
    L = oracle.layout(tp2, 944, False, 1 << 40, _lib=lib)
    assert L.check_backends(False, False) == 0
    L = oracle.layout(W.CONFIGS[1].layers, 944, False, 1 << 40, _lib=lib)
    assert L.check_backends(False, False) == oracle.BK_PADDED_ATTENTION
    assert L.check_backends(True, False) == 0
    L = oracle.layout(W.CONFIGS[1].layers, 944, True, 1 << 40, _lib=lib)
    assert L.check_backends(True, False) == oracle.BK_PACKED_STATE
    assert L.check_backends(False, False) == oracle.BK_PACKED_STATE | oracle.BK_PACKED_ATTENTION
    assert L.check_backends(True, True) == 0
    mla_only = [W.mla(1152), W.mla(656), W.mla(1152)]
    L = oracle.layout(mla_only, 64, True, 1 << 30, _lib=lib)
    assert L.check_backends(True, False) == 0 and L.check_backends(False, True) == oracle.BK_PACKED_ATTENTION
    # equal pages: nothing is padded, any backend reads the padded path
    L = oracle.layout([W.mla(1152), W.mla(1152)], 64, False, 1 << 30, _lib=lib)
    assert L.check_backends(False, False) == 0


def _brute_copies(B, pool, pairs, order):
    """The pairs applied by the brute force one after another ("forward",
    "reverse"), or all read before any is written ("together")."""
    out = pool.copy()
    if order == "together":
        for g, P in enumerate(pairs):
            for p in P:
                for i in B.groups[g]:
                    B.view(out, i)[int(p["dst_block"])] = B.view(pool, i)[int(p["src_block"])]
        return out
    seq = [(g, p) for g, P in enumerate(pairs) for p in P]
    for g, p in (seq if order == "forward" else seq[::-1]):
        brute.copy_blocks(B, out, [P if k == g else P[:0] for k, P in enumerate(pairs[:g])] +
                          [np.array([p], dtype=oracle.PAIR_DTYPE)] + [P[:0] for P in pairs[g + 1:]])
    return out


def check_copy_collisions(lib):
    """The pairs of one copy call run at the same time ("When Prefix Cache
    Meets KDA", Copy-on-Write: each hit its own private slot; Snapshot: each
    state its own spare buffer). Against the brute force: whenever the
    oracle accepts a batch, applying its pairs in any order (forward,
    reverse, all reads first) gives the oracle's result; whenever two orders
    give different pools, the oracle refuses the batch (OVERLAP) and writes
    nothing. Batches draw ids from a few blocks so collisions are common,
    across KV groups too (equal block ids share memory)."""
    rng = np.random.default_rng(29)
    refused = accepted = 0
    for t in range(80):
        spec = random_spec(rng, int(rng.integers(2, 7)))
        N = int(rng.choice([2, 4]))
        try:
            L = oracle.layout(spec, N, bool(t % 2), int(rng.integers(4000, 20000)), split_groups=bool(t % 3),
                              _lib=lib)
        except oracle.OracleError:
            continue
        if L.num_blocks < 3:
            continue
        B = brute.BruteLayout(spec, N, L.packed, L.pool_bytes, bool(t % 3))
        pool = W.fill_normal_np(L.pool_bytes, 100 + t)
        span = int(rng.integers(3, min(L.num_blocks, 8) + 1))
        pairs = []
        for g in range(L.num_kv_groups):
            k = int(rng.integers(0, 3))
            pairs.append(np.array([(int(rng.integers(0, span)), int(rng.integers(0, span))) for _ in range(k)],
                                  dtype=oracle.PAIR_DTYPE).reshape(-1))
        results = [_brute_copies(B, pool, pairs, o) for o in ("forward", "reverse", "together")]
        out = pool.copy()
        try:
            assert oracle.copy_blocks(L, out, pairs) == 0
        except oracle.OracleError as e:
            assert e.code == oracle.ERR_OVERLAP, e.code
            assert np.array_equal(out, pool), "a refused batch must copy nothing"
            refused += 1
            continue
        accepted += 1
        for r in results:
            assert np.array_equal(out, r), "an accepted batch depends on the order of its pairs"
    assert refused >= 10 and accepted >= 10, (refused, accepted)
    # order-dependent batches, planted: two pairs writing one block, a pair
    # writing a block another reads (in another KV group)
    L = oracle.layout(W.CONFIGS[0].layers, 64, False, 64 * 73_728, _lib=lib)
    B = brute.BruteLayout(W.CONFIGS[0].layers, 64, False, L.pool_bytes)
    pool = W.fill_normal_np(L.pool_bytes, 3)
    e0 = np.zeros(0, dtype=oracle.PAIR_DTYPE)
    for pairs in ([np.array([(1, 9), (2, 9)], dtype=oracle.PAIR_DTYPE), e0, e0, e0],
                  [np.array([(1, 9)], dtype=oracle.PAIR_DTYPE), e0, np.array([(9, 12)], dtype=oracle.PAIR_DTYPE), e0]):
        fw, rv = _brute_copies(B, pool, pairs, "forward"), _brute_copies(B, pool, pairs, "reverse")
        assert not np.array_equal(fw, rv)
        try:
            oracle.copy_blocks(L, pool.copy(), pairs)
            raise AssertionError("an order-dependent batch was accepted")
        except oracle.OracleError as e:
            assert e.code == oracle.ERR_OVERLAP


def _tagged_pool(B):
    """Every 4-byte word of every page of block b holds b (all layers)."""
    pool = np.full(B.pool_bytes, 0xEE, dtype=np.uint8)
    for i in range(len(B.spec)):
        v = B.view(pool, i)
        for b in range(B.num_blocks):
            v[b] = np.full(v[b].size // 4, b, dtype=np.int32).view(np.uint8).reshape(v[b].shape)
    return pool


def check_disjoint(lib):
    """The mixed step's guard against the brute force: on a pool whose pages
    are tagged with their block id, the blocks a chunk batch touches are the
    tags its objects pick up when the brute force stores them; the oracle's
    smallest common block of the load and the store side must be the
    smallest common tag (-1 when none), on the mixed workload's structure
    (KDA x3, SWA, MLA; chunk = 2N) and with shared blocks planted."""
    layers = []
    for _ in range(2):
        layers += [{"kind": "KDA", "token_bytes": 0, "conv_bytes": 16, "rec_bytes": 64, "window": 0}] * 3
        layers += [W.swa(16, 12), W.mla(16)]
    cfg = W.Config(600, "mixed-small", layers, N=4, requested_chunk=8, packed=True, num_requests=8,
                   lengths="fixed", fixed_lengths=(40, 23, 57, 31, 64, 17, 12, 48), snapshot="block", seed=6,
                   mixed=True)
    C = oracle.negotiate_chunk(8, 4, _lib=lib)
    inp = W.make_inputs(cfg, lambda mem: oracle.layout(layers, 4, True, mem, _lib=lib), C)
    L = inp.layout
    B = brute.BruteLayout(layers, 4, True, L.pool_bytes)
    pool = _tagged_pool(B)

    def tags(tables, jobs, nbytes):
        arena = np.full(nbytes, 0xFF, dtype=np.uint8)
        brute.store(B, C, pool, tables, jobs, arena)
        ids = np.unique(arena.view(np.int32))
        return set(int(x) for x in ids if x >= 0)

    rng = np.random.default_rng(6)
    store_side = sorted(tags(inp.tables_src, inp.store_jobs, inp.store_arena_bytes))
    seen_shared = 0
    for t in range(40):
        tables = [x.copy() for x in inp.tables_src]
        lj = [j.copy() for j in inp.load_jobs]
        if t > 0:
            # point one table entry at a block the store side reads (or at
            # any block): shared only if the load side uses that entry
            k = int(rng.integers(0, len(tables)))
            r, c = np.argwhere(tables[k] >= 0)[int(rng.integers(0, int((tables[k] >= 0).sum())))]
            pick = store_side if t % 3 else range(L.num_blocks)
            tables[k][r, c] = int(pick[int(rng.integers(0, len(pick)))])
        common = tags(tables, lj, inp.load_arena_bytes) & tags(tables, inp.store_jobs, inp.store_arena_bytes)
        want = min(common) if common else -1
        seen_shared += want >= 0
        assert oracle.check_disjoint(L, C, tables, lj, tables, inp.store_jobs) == want, (t, want)
    assert seen_shared >= 5
    # block-granular batches: the stored chunks as objects of m blocks from
    # their first block, KDA layers holding the last snapshot or every one;
    # the two sides are the even and the odd requests' stores (every block
    # position of those objects holds a block, as the brute force needs)
    m = C // 4

    def block_jobs(jobs, every, parity):
        units = [[(int(j["request"]), int(j["chunk"]) * m) for j in J if int(j["request"]) % 2 == parity]
                 for J in jobs]
        sizes = [L.object_bytes_blocks(m, every, g) for g in range(L.num_object_groups)]
        return W.pack_jobs(units, sizes)

    def block_tags(tables, jobs, nbytes, every):
        arena = np.full(nbytes, 0xFF, dtype=np.uint8)
        brute.store(B, C, pool, tables, jobs, arena, nb=m, kda_every=every)
        return set(int(x) for x in np.unique(arena.view(np.int32)) if x >= 0)

    kda_og = L.object_group[[l["kind"] for l in layers].index("KDA")]
    kda_kv = sorted({L.kv_group[i] for i in range(len(layers)) if layers[i]["kind"] == "KDA"})
    for every in (False, True):
        (aj, an), (bj, bn) = block_jobs(inp.store_jobs, every, 0), block_jobs(inp.store_jobs, every, 1)
        b_side = sorted(block_tags(inp.tables_src, bj, bn, every))
        hits = 0
        for t in range(16):
            tables = [x.copy() for x in inp.tables_src]
            if t % 2:
                # the first (not the last) KDA position of one even-request
                # object now holds a block the odd requests read
                job = aj[kda_og][int(rng.integers(0, len(aj[kda_og])))]
                k = kda_kv[int(rng.integers(0, len(kda_kv)))]
                tables[k][int(job["request"]), int(job["chunk"])] = b_side[int(rng.integers(0, len(b_side)))]
            elif t:
                k = int(rng.integers(0, len(tables)))
                r, c = np.argwhere(tables[k] >= 0)[int(rng.integers(0, int((tables[k] >= 0).sum())))]
                tables[k][r, c] = b_side[int(rng.integers(0, len(b_side)))]
            common = block_tags(tables, aj, an, every) & block_tags(tables, bj, bn, every)
            want = min(common) if common else -1
            hits += want >= 0
            got = oracle.check_disjoint(L, C, tables, aj, tables, bj, nb=m, kda_every=every)
            assert got == want, (every, t, got, want)
        assert hits >= (8 if every else 1), (every, hits)


ALL = ["check_negotiation_golden", "check_negotiation_bruteforce", "check_negotiation_edges",
       "check_budget", "check_page_formulas", "check_unified_block_size", "check_k3_groups", "check_closed_forms",
       "check_non_overlap", "check_store_load_cases", "check_block_objects", "check_copy_blocks",
       "check_copy_collisions", "check_disjoint",
       "check_q8_golden", "check_q8_random", "check_q8_objects", "check_q8_block_objects", "check_backends"]


def check_store_load_cases(lib):
    check_store_load(lib, tiny_case(lib, 0))
    rng = np.random.default_rng(11)
    for t in range(8):
        spec = random_spec(rng, int(rng.integers(2, 7)))
        spec[0] = W.mla(int(rng.choice([16, 32])))
        spec[-1] = {"kind": "KDA", "token_bytes": 0, "conv_bytes": 48, "rec_bytes": 256, "window": 0}
        N = int(rng.choice([2, 4]))
        lengths = [int(x) for x in rng.integers(N, 12 * N, size=3)]
        case = tiny_case(lib, spec=spec, N=N, req_chunk=int(rng.integers(1, 3 * N)),
                         packed=bool(t % 2), lengths=lengths, seed=t,
                         snapshot="block", split=bool((t // 2) % 2), separate=bool((t // 4) % 2 == 0))
        check_store_load(lib, case)
    check_errors(lib, tiny_case(lib, 0))


if __name__ == "__main__":
    handle = oracle.load_variant(sys.argv[1])
    for name in ALL:
        globals()[name](handle)
    print("all pins hold")

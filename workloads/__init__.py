"""Seeded synthetic inputs for the cache-paging workloads.

This module serves both the CUDA path's tests/benchmark and the oracle's
tests. It holds data (layer lists, sizes, seeds) and random draws only: it
computes no layout, no chunk negotiation and no page copy. Everything that
comes out of the layout (KV-group kinds, number of blocks, object sizes, the
negotiated chunk) is handed in by the caller.

Workload shapes follow the pages' deployments: Kimi-Linear (MLA latent 576
bf16 per token, KDA with 32 heads of d=128, conv window 3) and Kimi K3 (93
layers = 69 KDA + 24 MLA, N = 768, fp8 MLA cache). Values are N(0,1) float32
draws; the cached pages are byte-opaque to the store and load, so the value
distribution does not enter the computation.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

JOB_DTYPE = np.dtype([("request", "<i4"), ("chunk", "<i4"), ("offset", "<i8")])
SENTINEL = 0xA5
OBJECT_ALIGN = 16


def mla(token_bytes):
    return {"kind": "MLA", "token_bytes": token_bytes, "conv_bytes": 0, "rec_bytes": 0, "window": 0}


def swa(token_bytes, window):
    return {"kind": "SWA", "token_bytes": token_bytes, "conv_bytes": 0, "rec_bytes": 0, "window": window}


def kda(conv_dim, conv_width, heads, d, conv_elem=2, state_elem=4):
    # conv_state (conv_dim, k-1) and recurrent_state (heads, d, d)
    return {"kind": "KDA", "token_bytes": 0, "conv_bytes": conv_dim * conv_width * conv_elem,
            "rec_bytes": heads * d * d * state_elem, "window": 0}


@dataclass
class Config:
    index: int
    name: str
    layers: list
    N: int
    requested_chunk: int
    packed: bool
    num_requests: int
    lengths: str                 # "fixed" or "lognormal"
    fixed_lengths: tuple = ()
    snapshot: str = "block"      # "block": every block boundary; "chunk": chunk ends only
    pool_blocks: int | None = None   # None: exactly the blocks the batch needs
    seed: int = 0
    waves: int = 1               # requests are processed in this many waves
    mixed: bool = False          # concurrent load of hits + store of new chunks
    extra: dict = field(default_factory=dict)


def _kimi_linear_layers():
    # 24 layers, (KDA, KDA, KDA, MLA) x 6: 18 KDA + 6 MLA
    k = kda(12288, 3, 32, 128)
    return [mla(1152) if i % 4 == 3 else dict(k) for i in range(24)]


def _k3_layers():
    # 93 layers, 69 KDA + 24 MLA: MLA at every fourth layer and at the last
    k = kda(3 * 64 * 128, 3, 64, 128)
    return [mla(576) if (i % 4 == 3 or i == 92) else dict(k) for i in range(93)]


def _mixed_layers():
    # 30 layers, (KDA, KDA, KDA, SWA-4096, MLA) x 6
    k = kda(12288, 3, 32, 128)
    out = []
    for i in range(30):
        p = i % 5
        out.append(dict(k) if p < 3 else (swa(1152, 4096) if p == 3 else mla(1152)))
    return out


CONFIGS = {
    0: Config(0, "tiny: 4 layers (KDA,KDA,KDA,MLA), N=64, 2 requests (300, 517 tokens), padded",
              [kda(768, 3, 4, 64), kda(768, 3, 4, 64), kda(768, 3, 4, 64), mla(1152)],
              N=64, requested_chunk=100, packed=False, num_requests=2, lengths="fixed",
              fixed_lengths=(300, 517), snapshot="block", pool_blocks=64, seed=0, extra={"state_d": 64}),
    1: Config(1, "kimi-linear 24L (18 KDA + 6 MLA), N=944, 32 x 8192 tokens, padded, chunk=N",
              _kimi_linear_layers(), N=944, requested_chunk=944, packed=False, num_requests=32,
              lengths="fixed", fixed_lengths=(8192,) * 32, snapshot="block", seed=1),
    2: Config(2, "kimi-linear 24L packed, 64 lognormal requests (median 4096, 1k-32k), chunk=2N",
              _kimi_linear_layers(), N=944, requested_chunk=1888, packed=True, num_requests=64,
              lengths="lognormal", snapshot="block", seed=2),
    3: Config(3, "kimi-k3 93L (69 KDA + 24 MLA, fp8 MLA), N=768, chunk 1500->1536, 4 x 131072 tokens, padded",
              _k3_layers(), N=768, requested_chunk=1500, packed=False, num_requests=4,
              lengths="fixed", fixed_lengths=(131072,) * 4, snapshot="chunk", seed=3, waves=4),
    4: Config(4, "mixed step: 30L (KDA x3, SWA-4096, MLA) x 6, packed, 256 requests, hits load || new store",
              _mixed_layers(), N=944, requested_chunk=944, packed=True, num_requests=256,
              lengths="lognormal", snapshot="block", seed=4, mixed=True),
}


def state_row_elems(cfg: Config) -> int:
    """Values per row of the KDA recurrent state (heads, d, d): d."""
    return int(cfg.extra.get("state_d", 128))


def request_lengths(cfg: Config) -> np.ndarray:
    if cfg.lengths == "fixed":
        return np.array(cfg.fixed_lengths, dtype=np.int64)
    rng = np.random.default_rng(cfg.seed)
    x = rng.lognormal(mean=math.log(4096.0), sigma=1.0, size=cfg.num_requests)
    return np.clip(np.floor(x), 1024, 32768).astype(np.int64)


def hit_chunks(cfg: Config, lengths: np.ndarray, C: int) -> np.ndarray:
    """Cached whole chunks per request for the mixed step: floor(u * full), u ~ U[0,1]."""
    rng = np.random.default_rng(cfg.seed + 500)
    u = rng.random(lengths.size)
    full = lengths // C
    return np.floor(u * full).astype(np.int64)


# ----------------------------------------------------------------------------
# Block tables: which (KV group, request, block position) hold a block.
# ----------------------------------------------------------------------------

def needed_positions(cfg: Config, kind: str, L: int, N: int, C: int, hit: int | None = None):
    """Block positions a request of L tokens holds in a KV group of `kind`,
    as the engine would have allocated them.

    Paged attention holds one block per N tokens. A KDA group holds a
    snapshot where a scheduler step ended on a block boundary: every
    boundary (budget in [N, 2N)) or only every chunk end. In the mixed step a
    request with `hit` cached chunks holds: all attention blocks, SWA blocks
    from the window before the hit boundary onward, and KDA snapshots from
    the hit boundary's state onward.
    """
    nblk = -(-L // N)
    full_blocks = L // N
    interval = N if cfg.snapshot == "block" else C
    if kind == "MLA":
        return list(range(nblk))
    if kind == "SWA":
        if hit is None:
            return list(range(nblk))
        window = int(cfg.layers[[l["kind"] for l in cfg.layers].index("SWA")]["window"])
        # whole chunks that intersect the window before the hit boundary
        first = (max(0, hit * C - window) // C) * (C // N)
        return list(range(first, nblk))
    snaps = [p for p in range(full_blocks) if ((p + 1) * N) % interval == 0]
    if hit is None:
        return snaps
    keep_from = hit * C  # the state at the hit boundary and every later one
    return [p for p in snaps if (p + 1) * N >= keep_from]


def count_blocks(cfg, kv_group_kinds, lengths, N, C, hits=None):
    total = 0
    for kind in kv_group_kinds:
        for r, L in enumerate(lengths):
            total += len(needed_positions(cfg, kind, int(L), N, C, None if hits is None else int(hits[r])))
    return total


def block_tables(cfg, kv_group_kinds, lengths, N, C, num_blocks, seed, hits=None):
    """One int32 table [num_requests, max blocks per request] per KV group;
    -1 marks positions without a block. Block ids are a random permutation
    of the pool's blocks, so every page is distinct."""
    cols = int(max(-(-int(L) // N) for L in lengths))
    perm = np.random.default_rng(seed).permutation(num_blocks).astype(np.int32)
    tables = []
    k = 0
    for kind in kv_group_kinds:
        t = np.full((len(lengths), cols), -1, dtype=np.int32)
        for r, L in enumerate(lengths):
            pos = needed_positions(cfg, kind, int(L), N, C, None if hits is None else int(hits[r]))
            if k + len(pos) > num_blocks:
                raise ValueError("pool too small for the batch")
            t[r, pos] = perm[k:k + len(pos)]
            k += len(pos)
        tables.append(t)
    return tables


# ----------------------------------------------------------------------------
# Jobs: which objects to move, and where they sit in the arena.
# ----------------------------------------------------------------------------

def _round_up(x, a):
    return -(-x // a) * a


def pack_jobs(units_per_group, object_bytes):
    """units_per_group[og] = list of (request, chunk). Offsets are packed in
    (request, chunk, object group) order, each 16-byte aligned. Returns
    (list of JOB_DTYPE arrays, arena bytes)."""
    allu = sorted({(r, c) for u in units_per_group for (r, c) in u})
    members = [set(u) for u in units_per_group]
    out = [[] for _ in units_per_group]
    off = 0
    for (r, c) in allu:
        for og, m in enumerate(members):
            if (r, c) in m:
                out[og].append((r, c, off))
                off += _round_up(int(object_bytes[og]), OBJECT_ALIGN)
    jobs = [np.array(o, dtype=JOB_DTYPE) if o else np.zeros(0, dtype=JOB_DTYPE) for o in out]
    return jobs, off


def store_units(lengths, C, num_object_groups, first_request=0):
    """Every whole chunk of every request, in every object group."""
    u = [(first_request + r, c) for r, L in enumerate(lengths) for c in range(int(L) // C)]
    return [list(u) for _ in range(num_object_groups)]


def mixed_units(cfg, lengths, hits, C, object_group_kinds):
    """Mixed step: load units (hits) and store units (new chunks) per object group."""
    window = int(next(l["window"] for l in cfg.layers if l["kind"] == "SWA"))
    load = [[] for _ in object_group_kinds]
    store = [[] for _ in object_group_kinds]
    for r, L in enumerate(lengths):
        full = int(L) // C
        h = int(hits[r])
        for og, kind in enumerate(object_group_kinds):
            if kind == "MLA":
                load[og] += [(r, c) for c in range(h)]
            elif kind == "SWA":
                lo = max(0, h * C - window)
                load[og] += [(r, c) for c in range(h) if (c + 1) * C > lo]
            else:
                if h > 0:
                    load[og].append((r, h - 1))
            store[og] += [(r, c) for c in range(h, full)]
    return load, store


# ----------------------------------------------------------------------------
# Byte content
# ----------------------------------------------------------------------------

def fill_normal(t, seed: int):
    """Fill a torch uint8 tensor with N(0,1) float32 draws (device-seeded)."""
    import torch
    g = torch.Generator(device=t.device)
    g.manual_seed(int(seed))
    n4 = (t.numel() // 4) * 4
    if n4:
        t[:n4].view(torch.float32).normal_(generator=g)
    if n4 < t.numel():
        t[n4:].random_(0, 256, generator=g)
    return t


def fill_normal_np(n: int, seed: int) -> np.ndarray:
    """N(0,1) float32 draws as a uint8 numpy buffer of n bytes (CPU-only tests)."""
    rng = np.random.default_rng(seed)
    buf = np.empty(n, dtype=np.uint8)
    n4 = (n // 4) * 4
    buf[:n4] = rng.standard_normal(n4 // 4, dtype=np.float32).view(np.uint8)
    buf[n4:] = rng.integers(0, 256, n - n4, dtype=np.uint8)
    return buf


def fill_normal_host(n: int, seed: int, threads: int = 1) -> np.ndarray:
    """N(0,1) float32 draws as a uint8 numpy buffer of n bytes, drawn by
    `threads` workers, each filling one contiguous part from its own stream
    of one seed sequence (for host-side runs over many GB)."""
    from concurrent.futures import ThreadPoolExecutor
    buf = np.empty(n, dtype=np.uint8)
    n4 = (n // 4) * 4
    f = buf[:n4].view(np.float32)
    k = max(1, int(threads))
    bounds = [f.size * i // k for i in range(k + 1)]
    streams = np.random.SeedSequence(int(seed)).spawn(k)

    def fill(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi > lo:
            np.random.default_rng(streams[i]).standard_normal(hi - lo, dtype=np.float32, out=f[lo:hi])
    with ThreadPoolExecutor(k) as ex:
        list(ex.map(fill, range(k)))
    buf[n4:] = np.random.default_rng(int(seed)).integers(0, 256, n - n4, dtype=np.uint8)
    return buf


# ----------------------------------------------------------------------------
# A whole batch of inputs for one workload
# ----------------------------------------------------------------------------

@dataclass
class Inputs:
    cfg: Config
    C: int
    layout: object
    request_ids: list
    lengths: np.ndarray
    object_bytes: list
    tables_src: list                  # store-side pool (and the mixed step's single pool)
    tables_dst: list | None = None    # load-side fresh pool
    jobs: list | None = None          # store jobs, also loaded back
    arena_bytes: int = 0
    hits: np.ndarray | None = None
    load_jobs: list | None = None     # mixed step
    load_arena_bytes: int = 0
    store_jobs: list | None = None
    store_arena_bytes: int = 0

    @property
    def payload_bytes(self):
        """Bytes of objects moved by one store (or one load) of `jobs`."""
        if self.jobs is None:
            return 0
        return sum(int(self.object_bytes[g]) * len(j) for g, j in enumerate(self.jobs))


def make_inputs(cfg: Config, build_layout, C: int, request_ids=None) -> Inputs:
    """Seeded inputs for `cfg`. `build_layout(mem_bytes)` builds the layout
    under test (oracle or library) and `C` is the negotiated chunk; the pool
    gets exactly the blocks the batch needs (or the workload's fixed count)."""
    all_lengths = request_lengths(cfg)
    ids = list(range(cfg.num_requests)) if request_ids is None else list(request_ids)
    lengths = all_lengths[ids]
    probe = build_layout(1 << 60)
    per_block = probe.pool_bytes // probe.num_blocks
    hits = hit_chunks(cfg, all_lengths, C)[ids] if cfg.mixed else None
    need = count_blocks(cfg, probe.kv_group_kind, lengths, cfg.N, C, hits)
    nb = cfg.pool_blocks or need
    layout = build_layout(nb * per_block)
    assert layout.num_blocks == nb
    sizes = [layout.object_bytes(C, g) for g in range(layout.num_object_groups)]
    seed = cfg.seed + 7919 * (ids[0] if ids else 0)
    src = block_tables(cfg, layout.kv_group_kind, lengths, cfg.N, C, nb, seed, hits)
    inp = Inputs(cfg=cfg, C=C, layout=layout, request_ids=ids, lengths=lengths, object_bytes=sizes,
                 tables_src=src, hits=hits)
    if cfg.mixed:
        og_kinds = [cfg.layers[layout.object_group.index(g)]["kind"] for g in range(layout.num_object_groups)]
        lu, su = mixed_units(cfg, lengths, hits, C, og_kinds)
        inp.load_jobs, inp.load_arena_bytes = pack_jobs(lu, sizes)
        inp.store_jobs, inp.store_arena_bytes = pack_jobs(su, sizes)
    else:
        inp.tables_dst = block_tables(cfg, layout.kv_group_kind, lengths, cfg.N, C, nb, seed + 1000)
        inp.jobs, inp.arena_bytes = pack_jobs(store_units(lengths, C, layout.num_object_groups), sizes)
    return inp

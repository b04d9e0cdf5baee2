"""CPU oracle for paging a hybrid KDA + MLA cache (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product library (``state_cache_paging_gb300``)
never imports it and shares no code with it.

Two independent implementations live here:

* ``oracle.c`` (loaded through ctypes): layout, chunk negotiation, the
  scheduler-budget rule, store and load, with explicit per-page address
  arithmetic and ``memcpy``.
* ``brute.py``: a numpy restatement that builds the per-layer views the way
  the vLLM blog describes them and gathers objects token by token.

Layer specs are plain dicts ``{"kind": "MLA"|"KDA"|"SWA", "token_bytes": int,
"conv_bytes": int, "rec_bytes": int, "window": int}``; jobs are numpy arrays of
``JOB_DTYPE`` (request int32, chunk int32, offset int64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle.h")]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

MAX_LAYERS = 256
KINDS = {"MLA": 0, "KDA": 1, "SWA": 2}
KIND_NAMES = {v: k for k, v in KINDS.items()}

OK = 0
ERR_INVALID_ARG = -1
ERR_ALIGN = -2
ERR_NOT_MULTIPLE = -3
ERR_NO_MEMORY = -4
ERR_OVERFLOW = -6
ERR_BUDGET = -7
ERR_OVERLAP = -8

ST_BLOCK_OOR = 0x1
ST_NO_BLOCK = 0x2
ST_NO_SNAPSHOT = 0x4
ST_BAD_JOB = 0x8

BK_PADDED_ATTENTION = 0x1
BK_PACKED_ATTENTION = 0x2
BK_PACKED_STATE = 0x4

JOB_DTYPE = np.dtype([("request", "<i4"), ("chunk", "<i4"), ("offset", "<i8")])


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle error {code}")
        self.code = code


def build(force: bool = False, out_path: str | None = None, src_path: str | None = None) -> str:
    """Compile oracle.c into a shared library with gcc; returns its path."""
    out = out_path or _LIB_PATH
    src = src_path or _SRC[0]
    stale = force or not os.path.exists(out) or any(
        os.path.getmtime(s) > os.path.getmtime(out) for s in _SRC if os.path.exists(s))
    if out_path is not None or stale:
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Werror",
                        "-I", _HERE, src, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, out)
    return out


class _Layer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32),
                ("token_bytes", ctypes.c_int64), ("conv_bytes", ctypes.c_int64),
                ("rec_bytes", ctypes.c_int64)]


_I32A = ctypes.c_int32 * MAX_LAYERS
_I64A = ctypes.c_int64 * MAX_LAYERS


class _Layout(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("packed", ctypes.c_int32),
                ("split_groups", ctypes.c_int32), ("separate_object_groups", ctypes.c_int32),
                ("N", ctypes.c_int64), ("mem_bytes", ctypes.c_int64),
                ("layers", _Layer * MAX_LAYERS),
                ("num_kv_groups", ctypes.c_int32), ("num_object_groups", ctypes.c_int32),
                ("num_slabs", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("page_size", ctypes.c_int64), ("block_stride", ctypes.c_int64),
                ("num_blocks", ctypes.c_int64), ("pool_bytes", ctypes.c_int64),
                ("kv_group", _I32A), ("slot", _I32A), ("object_group", _I32A),
                ("kv_group_kind", _I32A), ("kv_group_size", _I32A),
                ("real_bytes", _I64A), ("page_bytes", _I64A),
                ("base", _I64A), ("stride", _I64A)]


class _Job(ctypes.Structure):
    _fields_ = [("request", ctypes.c_int32), ("chunk", ctypes.c_int32), ("offset", ctypes.c_int64)]


class _Tables(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("num_kv_groups", ctypes.c_int32),
                ("table", ctypes.POINTER(ctypes.POINTER(ctypes.c_int32))),
                ("row_stride", ctypes.POINTER(ctypes.c_int64)),
                ("num_cols", ctypes.POINTER(ctypes.c_int64))]


class _Page(ctypes.Structure):
    _fields_ = [("pool_offset", ctypes.c_int64), ("object_offset", ctypes.c_int64), ("bytes", ctypes.c_int64),
                ("layer", ctypes.c_int32), ("block", ctypes.c_int32)]


PAGE_DTYPE = np.dtype([("pool_offset", "<i8"), ("object_offset", "<i8"), ("bytes", "<i8"),
                       ("layer", "<i4"), ("block", "<i4")])
assert PAGE_DTYPE.itemsize == ctypes.sizeof(_Page)  # the C oracle fills or_page records in place


class _PageList(ctypes.Structure):
    _fields_ = [("pages", ctypes.c_void_p), ("capacity", ctypes.c_int64), ("count", ctypes.c_int64)]


class _Pair(ctypes.Structure):
    _fields_ = [("src_block", ctypes.c_int32), ("dst_block", ctypes.c_int32)]


PAIR_DTYPE = np.dtype([("src_block", "<i4"), ("dst_block", "<i4")])


class _CopyBatch(ctypes.Structure):
    _fields_ = [("num_kv_groups", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("pairs", ctypes.POINTER(ctypes.POINTER(_Pair))), ("num_pairs", ctypes.POINTER(ctypes.c_int64))]


class _Jobs(ctypes.Structure):
    _fields_ = [("num_object_groups", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("jobs", ctypes.POINTER(ctypes.POINTER(_Job))),
                ("num_jobs", ctypes.POINTER(ctypes.c_int64))]


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.POINTER
    lib.or_negotiate_chunk.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P(ctypes.c_int64)]
    lib.or_check_step_budget.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    lib.or_layout_build.argtypes = [P(_Layout)]
    lib.or_object_bytes.argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_int]
    lib.or_object_bytes.restype = ctypes.c_int64
    for name in ("or_store", "or_load"):
        getattr(lib, name).argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_void_p, P(_Tables),
                                       P(_Jobs), ctypes.c_void_p, ctypes.c_int64, P(ctypes.c_uint32)]
    lib.or_list_pages.argtypes = [P(_Layout), ctypes.c_int64, P(_Tables), P(_Jobs), ctypes.c_int64,
                                  P(ctypes.c_uint32), P(_PageList)]
    lib.or_list_pages_any.argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P(_Tables),
                                      P(_Jobs), ctypes.c_int64, P(ctypes.c_uint32), P(_PageList)]
    lib.or_object_bytes_blocks.argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    lib.or_object_bytes_blocks.restype = ctypes.c_int64
    for name in ("or_store_blocks", "or_load_blocks"):
        getattr(lib, name).argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, P(_Tables),
                                       P(_Jobs), ctypes.c_void_p, ctypes.c_int64, P(ctypes.c_uint32)]
    lib.or_check_backends.argtypes = [P(_Layout), ctypes.c_int, ctypes.c_int]
    lib.or_check_backends.restype = ctypes.c_uint32
    lib.or_copy_blocks.argtypes = [P(_Layout), ctypes.c_void_p, P(_CopyBatch), P(ctypes.c_uint32)]
    lib.or_check_disjoint.argtypes = [P(_Layout), ctypes.c_int64, P(_Tables), P(_Jobs), P(_Tables), P(_Jobs),
                                      P(ctypes.c_int32)]
    lib.or_check_disjoint_blocks.argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_int, P(_Tables), P(_Jobs),
                                             P(_Tables), P(_Jobs), P(ctypes.c_int32)]
    for name in ("or_store_q8", "or_load_q8"):
        getattr(lib, name).argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, P(_Tables),
                                       P(_Jobs), ctypes.c_void_p, ctypes.c_int64, P(ctypes.c_uint32)]
    lib.or_object_bytes_q8.argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    lib.or_object_bytes_q8.restype = ctypes.c_int64
    for name in ("or_store_blocks_q8", "or_load_blocks_q8"):
        getattr(lib, name).argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                       P(_Tables), P(_Jobs), ctypes.c_void_p, ctypes.c_int64, P(ctypes.c_uint32)]
    lib.or_object_bytes_blocks_q8.argtypes = [P(_Layout), ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_int]
    lib.or_object_bytes_blocks_q8.restype = ctypes.c_int64
    lib.or_unified_block_size.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P(ctypes.c_int64)]
    return lib


_lib: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def load_variant(path: str) -> ctypes.CDLL:
    """Load another build of the oracle (used by the mutation tests)."""
    return _bind(ctypes.CDLL(path))


# ----------------------------------------------------------------------------
# Negotiation and budget
# ----------------------------------------------------------------------------

def negotiate_chunk(requested: int, N: int, strict: bool = False, _lib=None) -> int:
    out = ctypes.c_int64(0)
    rc = (_lib or lib()).or_negotiate_chunk(int(requested), int(N), int(bool(strict)), ctypes.byref(out))
    if rc != OK:
        raise OracleError(rc, f"negotiate_chunk({requested}, {N}, strict={strict})")
    return out.value


def unified_block_size(attn_token_bytes: int, state_page_bytes: int, align: int = 16, _lib=None) -> int:
    out = ctypes.c_int64(0)
    rc = (_lib or lib()).or_unified_block_size(int(attn_token_bytes), int(state_page_bytes), int(align),
                                               ctypes.byref(out))
    if rc != OK:
        raise OracleError(rc, "unified_block_size")
    return out.value


def check_step_budget(N: int, max_batched: int, separate_object_groups: bool, _lib=None) -> int:
    """Returns the oracle's code: 0 when the budget is allowed."""
    return (_lib or lib()).or_check_step_budget(int(N), int(max_batched), int(bool(separate_object_groups)))


# ----------------------------------------------------------------------------
# Layout
# ----------------------------------------------------------------------------

@dataclass
class Layout:
    """The oracle's layout, as plain Python values."""
    N: int
    packed: bool
    num_kv_groups: int
    num_object_groups: int
    num_slabs: int
    page_size: int
    block_stride: int
    num_blocks: int
    pool_bytes: int
    kv_group: list
    slot: list
    object_group: list
    kv_group_kind: list
    kv_group_size: list
    real_bytes: list
    page_bytes: list
    base: list
    stride: list
    kinds: list
    _c: _Layout = field(repr=False, default=None)
    _lib: object = field(repr=False, default=None)

    def object_bytes(self, C: int, og: int) -> int:
        return int(self._lib.or_object_bytes(ctypes.byref(self._c), int(C), int(og)))

    def check_backends(self, attn_indexes_by_stride: bool, state_pages_strided_ok: bool) -> int:
        return int(self._lib.or_check_backends(ctypes.byref(self._c), int(bool(attn_indexes_by_stride)),
                                               int(bool(state_pages_strided_ok))))

    def object_bytes_q8(self, C: int, d: int, og: int) -> int:
        return int(self._lib.or_object_bytes_q8(ctypes.byref(self._c), int(C), int(d), int(og)))

    def object_bytes_blocks(self, nb: int, kda_every: bool, og: int) -> int:
        return int(self._lib.or_object_bytes_blocks(ctypes.byref(self._c), int(nb), int(bool(kda_every)), int(og)))

    def object_bytes_blocks_q8(self, nb: int, kda_every: bool, d: int, og: int) -> int:
        return int(self._lib.or_object_bytes_blocks_q8(ctypes.byref(self._c), int(nb), int(bool(kda_every)), int(d),
                                                       int(og)))


def _fill_layout(spec_layers, N, packed, mem_bytes, split_groups, separate_object_groups) -> _Layout:
    if len(spec_layers) > MAX_LAYERS:
        raise OracleError(ERR_INVALID_ARG, "too many layers")
    c = _Layout()
    c.num_layers = len(spec_layers)
    c.packed = int(bool(packed))
    c.split_groups = int(bool(split_groups))
    c.separate_object_groups = int(bool(separate_object_groups))
    c.N = int(N)
    c.mem_bytes = int(mem_bytes)
    for i, l in enumerate(spec_layers):
        c.layers[i].kind = KINDS[l["kind"]]
        c.layers[i].window = int(l.get("window", 0))
        c.layers[i].token_bytes = int(l.get("token_bytes", 0))
        c.layers[i].conv_bytes = int(l.get("conv_bytes", 0))
        c.layers[i].rec_bytes = int(l.get("rec_bytes", 0))
    return c


def layout(spec_layers, N, packed, mem_bytes, split_groups=True, separate_object_groups=True,
           _lib=None) -> Layout:
    lb = _lib or lib()
    c = _fill_layout(spec_layers, N, packed, mem_bytes, split_groups, separate_object_groups)
    rc = lb.or_layout_build(ctypes.byref(c))
    if rc != OK:
        raise OracleError(rc, "layout_build")
    n = c.num_layers
    g = c.num_kv_groups
    return Layout(
        N=c.N, packed=bool(c.packed), num_kv_groups=g, num_object_groups=c.num_object_groups,
        num_slabs=c.num_slabs, page_size=c.page_size, block_stride=c.block_stride,
        num_blocks=c.num_blocks, pool_bytes=c.pool_bytes,
        kv_group=list(c.kv_group[:n]), slot=list(c.slot[:n]), object_group=list(c.object_group[:n]),
        kv_group_kind=[KIND_NAMES[k] for k in c.kv_group_kind[:g]],
        kv_group_size=list(c.kv_group_size[:g]),
        real_bytes=list(c.real_bytes[:n]), page_bytes=list(c.page_bytes[:n]),
        base=list(c.base[:n]), stride=list(c.stride[:n]),
        kinds=[l["kind"] for l in spec_layers], _c=c, _lib=lb)


# ----------------------------------------------------------------------------
# Store / load
# ----------------------------------------------------------------------------

def _marshal(L: Layout, tables, jobs):
    keep = []
    g = L.num_kv_groups
    if len(tables) != g:
        raise OracleError(ERR_INVALID_ARG, "one block table per KV group is required")
    nreq = tables[0].shape[0] if g else 0
    tptrs = (ctypes.POINTER(ctypes.c_int32) * g)()
    strides = (ctypes.c_int64 * g)()
    cols = (ctypes.c_int64 * g)()
    for k, t in enumerate(tables):
        t = np.ascontiguousarray(t, dtype=np.int32)
        if t.ndim != 2 or t.shape[0] != nreq:
            raise OracleError(ERR_INVALID_ARG, "block tables must be [num_requests, cols]")
        keep.append(t)
        tptrs[k] = t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        strides[k] = t.shape[1]
        cols[k] = t.shape[1]
    T = _Tables(num_requests=nreq, num_kv_groups=g, table=tptrs, row_stride=strides, num_cols=cols)
    o = L.num_object_groups
    if len(jobs) != o:
        raise OracleError(ERR_INVALID_ARG, "one job array per object group is required")
    jptrs = (ctypes.POINTER(_Job) * o)()
    counts = (ctypes.c_int64 * o)()
    for q, j in enumerate(jobs):
        j = np.ascontiguousarray(j, dtype=JOB_DTYPE)
        keep.append(j)
        jptrs[q] = j.ctypes.data_as(ctypes.POINTER(_Job))
        counts[q] = j.shape[0]
    J = _Jobs(num_object_groups=o, jobs=jptrs, num_jobs=counts)
    keep += [tptrs, strides, cols, jptrs, counts]
    return T, J, keep


def store(L: Layout, C: int, pool: np.ndarray, tables, jobs, arena: np.ndarray) -> int:
    """Gathers objects from ``pool`` into ``arena``; returns the status bits."""
    assert pool.dtype == np.uint8 and arena.dtype == np.uint8
    assert pool.flags.c_contiguous and arena.flags.c_contiguous and arena.flags.writeable
    if pool.size < L.pool_bytes:
        raise OracleError(ERR_INVALID_ARG, "pool smaller than the layout")
    T, J, keep = _marshal(L, tables, jobs)
    st = ctypes.c_uint32(0)
    rc = L._lib.or_store(ctypes.byref(L._c), int(C), pool.ctypes.data, ctypes.byref(T), ctypes.byref(J),
                         arena.ctypes.data, arena.size, ctypes.byref(st))
    if rc != OK:
        raise OracleError(rc, "store")
    return st.value


def load(L: Layout, C: int, pool: np.ndarray, tables, jobs, arena: np.ndarray) -> int:
    """Scatters objects from ``arena`` into ``pool``; returns the status bits."""
    assert pool.dtype == np.uint8 and arena.dtype == np.uint8
    assert pool.flags.c_contiguous and arena.flags.c_contiguous and pool.flags.writeable
    if pool.size < L.pool_bytes:
        raise OracleError(ERR_INVALID_ARG, "pool smaller than the layout")
    T, J, keep = _marshal(L, tables, jobs)
    st = ctypes.c_uint32(0)
    rc = L._lib.or_load(ctypes.byref(L._c), int(C), pool.ctypes.data, ctypes.byref(T), ctypes.byref(J),
                        arena.ctypes.data, arena.size, ctypes.byref(st))
    if rc != OK:
        raise OracleError(rc, "load")
    return st.value


def store_blocks(L: Layout, nb: int, kda_every: bool, pool: np.ndarray, tables, jobs, arena: np.ndarray) -> int:
    """Block-granular store: each job's `chunk` field is its first block
    position; every object covers `nb` blocks. Returns the status bits."""
    assert pool.dtype == np.uint8 and arena.dtype == np.uint8 and arena.flags.writeable
    T, J, keep = _marshal(L, tables, jobs)
    st = ctypes.c_uint32(0)
    rc = L._lib.or_store_blocks(ctypes.byref(L._c), int(nb), int(bool(kda_every)), pool.ctypes.data,
                                ctypes.byref(T), ctypes.byref(J), arena.ctypes.data, arena.size, ctypes.byref(st))
    if rc != OK:
        raise OracleError(rc, "store_blocks")
    return st.value


def load_blocks(L: Layout, nb: int, kda_every: bool, pool: np.ndarray, tables, jobs, arena: np.ndarray) -> int:
    assert pool.dtype == np.uint8 and arena.dtype == np.uint8 and pool.flags.writeable
    T, J, keep = _marshal(L, tables, jobs)
    st = ctypes.c_uint32(0)
    rc = L._lib.or_load_blocks(ctypes.byref(L._c), int(nb), int(bool(kda_every)), pool.ctypes.data,
                               ctypes.byref(T), ctypes.byref(J), arena.ctypes.data, arena.size, ctypes.byref(st))
    if rc != OK:
        raise OracleError(rc, "load_blocks")
    return st.value


def store_q8(L: Layout, C: int, d: int, pool: np.ndarray, tables, jobs, arena: np.ndarray) -> int:
    """Chunk-form store with INT8 records for the KDA recurrent state
    (rows of d fp32 values). Returns the status bits."""
    assert pool.dtype == np.uint8 and arena.dtype == np.uint8 and arena.flags.writeable
    T, J, keep = _marshal(L, tables, jobs)
    st = ctypes.c_uint32(0)
    rc = L._lib.or_store_q8(ctypes.byref(L._c), int(C), int(d), pool.ctypes.data, ctypes.byref(T),
                            ctypes.byref(J), arena.ctypes.data, arena.size, ctypes.byref(st))
    if rc != OK:
        raise OracleError(rc, "store_q8")
    return st.value


def load_q8(L: Layout, C: int, d: int, pool: np.ndarray, tables, jobs, arena: np.ndarray) -> int:
    assert pool.dtype == np.uint8 and arena.dtype == np.uint8 and pool.flags.writeable
    T, J, keep = _marshal(L, tables, jobs)
    st = ctypes.c_uint32(0)
    rc = L._lib.or_load_q8(ctypes.byref(L._c), int(C), int(d), pool.ctypes.data, ctypes.byref(T),
                           ctypes.byref(J), arena.ctypes.data, arena.size, ctypes.byref(st))
    if rc != OK:
        raise OracleError(rc, "load_q8")
    return st.value


def store_blocks_q8(L: Layout, nb: int, kda_every: bool, d: int, pool: np.ndarray, tables, jobs,
                    arena: np.ndarray) -> int:
    """Block-granular store with INT8 records for every stored KDA snapshot.
    Returns the status bits."""
    assert pool.dtype == np.uint8 and arena.dtype == np.uint8 and arena.flags.writeable
    T, J, keep = _marshal(L, tables, jobs)
    st = ctypes.c_uint32(0)
    rc = L._lib.or_store_blocks_q8(ctypes.byref(L._c), int(nb), int(bool(kda_every)), int(d), pool.ctypes.data,
                                   ctypes.byref(T), ctypes.byref(J), arena.ctypes.data, arena.size,
                                   ctypes.byref(st))
    if rc != OK:
        raise OracleError(rc, "store_blocks_q8")
    return st.value


def load_blocks_q8(L: Layout, nb: int, kda_every: bool, d: int, pool: np.ndarray, tables, jobs,
                   arena: np.ndarray) -> int:
    assert pool.dtype == np.uint8 and arena.dtype == np.uint8 and pool.flags.writeable
    T, J, keep = _marshal(L, tables, jobs)
    st = ctypes.c_uint32(0)
    rc = L._lib.or_load_blocks_q8(ctypes.byref(L._c), int(nb), int(bool(kda_every)), int(d), pool.ctypes.data,
                                  ctypes.byref(T), ctypes.byref(J), arena.ctypes.data, arena.size,
                                  ctypes.byref(st))
    if rc != OK:
        raise OracleError(rc, "load_blocks_q8")
    return st.value


def copy_blocks(L: Layout, pool: np.ndarray, pairs) -> int:
    """In-pool copies: pairs[g] is a PAIR_DTYPE array for KV group g."""
    assert pool.dtype == np.uint8 and pool.flags.writeable and pool.size >= L.pool_bytes
    g = L.num_kv_groups
    if len(pairs) != g:
        raise OracleError(ERR_INVALID_ARG, "one pair array per KV group is required")
    ptrs = (ctypes.POINTER(_Pair) * g)()
    counts = (ctypes.c_int64 * g)()
    keep = []
    for k, p in enumerate(pairs):
        p = np.ascontiguousarray(p, dtype=PAIR_DTYPE)
        keep.append(p)
        ptrs[k] = p.ctypes.data_as(ctypes.POINTER(_Pair))
        counts[k] = p.shape[0]
    B = _CopyBatch(num_kv_groups=g, pairs=ptrs, num_pairs=counts)
    st = ctypes.c_uint32(0)
    rc = L._lib.or_copy_blocks(ctypes.byref(L._c), pool.ctypes.data, ctypes.byref(B), ctypes.byref(st))
    if rc != OK:
        raise OracleError(rc, "copy_blocks")
    return st.value


def check_disjoint(L: Layout, C: int, tables_a, jobs_a, tables_b, jobs_b, nb: int = 0,
                   kda_every: bool = False) -> int:
    """-1 when the chunk batches (tables_a, jobs_a) and (tables_b, jobs_b)
    touch disjoint blocks, else the smallest block both touch. nb > 0
    selects the block-granular form (C is then ignored)."""
    Ta, Ja, keep_a = _marshal(L, tables_a, jobs_a)
    Tb, Jb, keep_b = _marshal(L, tables_b, jobs_b)
    out = ctypes.c_int32(0)
    if nb:
        rc = L._lib.or_check_disjoint_blocks(ctypes.byref(L._c), int(nb), int(bool(kda_every)), ctypes.byref(Ta),
                                             ctypes.byref(Ja), ctypes.byref(Tb), ctypes.byref(Jb), ctypes.byref(out))
    else:
        rc = L._lib.or_check_disjoint(ctypes.byref(L._c), int(C), ctypes.byref(Ta), ctypes.byref(Ja),
                                      ctypes.byref(Tb), ctypes.byref(Jb), ctypes.byref(out))
    if rc == ERR_OVERLAP:
        return out.value
    if rc != OK:
        raise OracleError(rc, "check_disjoint")
    return -1


def list_pages(L: Layout, C: int, tables, jobs, arena_bytes: int, nb: int = 0, kda_every: bool = False):
    """The pages a store/load of `jobs` touches, as a PAGE_DTYPE array
    (pool offset, arena offset, bytes, layer, block), plus the status bits.
    nb > 0 selects the block-granular form (C is then ignored)."""
    T, J, keep = _marshal(L, tables, jobs)

    def run(pl):
        st = ctypes.c_uint32(0)
        rc = L._lib.or_list_pages_any(ctypes.byref(L._c), int(C), int(nb), int(bool(kda_every)), ctypes.byref(T),
                                      ctypes.byref(J), int(arena_bytes), ctypes.byref(st), ctypes.byref(pl))
        if rc != OK:
            raise OracleError(rc, "list_pages")
        return st.value

    pl = _PageList(None, 0, 0)
    run(pl)
    out = np.zeros(pl.count, dtype=PAGE_DTYPE)
    pl = _PageList(out.ctypes.data, out.size, 0)
    st = run(pl)
    assert pl.count == out.size
    return out, st

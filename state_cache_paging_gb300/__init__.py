"""state_cache_paging_gb300 -- paging a hybrid KDA + MLA model's cache between
a vLLM-style paged GPU pool and LMCache-style per-chunk objects on GB300.

A thin ctypes binding over ``liblmc.so`` (C ABI in ``include/lmc.h``). The
Python functions carry the C names and only marshal arguments: the layout,
negotiation and budget rules run in the library's host code, and every byte
of a store or load is moved by the library's sm_103a kernels. PyTorch is used
for device memory and streams only.

Importing this package raises ImportError when ``liblmc.so`` has not been
built (``python state_cache_paging_gb300/build.py``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblmc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"liblmc.so is not built at {LIB_PATH}: run `python state_cache_paging_gb300/build.py`")

_lib = None  # bound by _use_library below

LMC_OK = 0
LMC_ERR_INVALID_ARG = -1
LMC_ERR_ALIGN = -2
LMC_ERR_NOT_MULTIPLE = -3
LMC_ERR_NO_MEMORY = -4
LMC_ERR_CUDA = -5
LMC_ERR_OVERFLOW = -6
LMC_ERR_BUDGET = -7
LMC_ERR_OVERLAP = -8

LMC_ST_BLOCK_OOR = 0x1
LMC_ST_NO_BLOCK = 0x2
LMC_ST_NO_SNAPSHOT = 0x4
LMC_ST_BAD_JOB = 0x8
LMC_ST_TIMEOUT = 0x10

LMC_BK_PADDED_ATTENTION = 0x1
LMC_BK_PACKED_ATTENTION = 0x2
LMC_BK_PACKED_STATE = 0x4

LMC_KDA_LAST_BLOCK = 0
LMC_KDA_EVERY_BLOCK = 1

LMC_LAYER = {"MLA": 0, "KDA": 1, "SWA": 2}
LMC_LAYER_NAME = {v: k for k, v in LMC_LAYER.items()}
LMC_MAX_LAYERS = 256

# An lmc_job record: request int32, chunk int32, arena offset int64.
JOB_DTYPE = np.dtype([("request", "<i4"), ("chunk", "<i4"), ("offset", "<i8")])
# An lmc_block_pair record: source block int32, destination block int32.
PAIR_DTYPE = np.dtype([("src_block", "<i4"), ("dst_block", "<i4")])


class LmcError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {lmc_strerror(code)}")
        self.code = code


class lmc_layer_spec(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32), ("token_bytes", ctypes.c_int64),
                ("conv_bytes", ctypes.c_int64), ("rec_bytes", ctypes.c_int64)]


class lmc_layout_params(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("mode", ctypes.c_int32), ("grouping", ctypes.c_int32),
                ("separate_object_groups", ctypes.c_int32), ("block_size", ctypes.c_int64),
                ("mem_bytes", ctypes.c_int64), ("layers", ctypes.POINTER(lmc_layer_spec))]


class lmc_layer_desc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("kv_group", ctypes.c_int32), ("slot", ctypes.c_int32),
                ("object_group", ctypes.c_int32), ("real_bytes", ctypes.c_int64),
                ("page_bytes", ctypes.c_int64), ("base", ctypes.c_int64), ("stride", ctypes.c_int64)]


class lmc_layout_info(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_kv_groups", ctypes.c_int32),
                ("num_object_groups", ctypes.c_int32), ("num_slabs", ctypes.c_int32),
                ("block_size", ctypes.c_int64), ("page_size", ctypes.c_int64),
                ("block_stride", ctypes.c_int64), ("num_blocks", ctypes.c_int64),
                ("pool_bytes", ctypes.c_int64), ("layers", ctypes.POINTER(lmc_layer_desc)),
                ("kv_group_kind", ctypes.POINTER(ctypes.c_int32)),
                ("kv_group_size", ctypes.POINTER(ctypes.c_int32)),
                ("object_group_kind", ctypes.POINTER(ctypes.c_int32))]


class lmc_block_table(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("row_stride", ctypes.c_int64), ("num_cols", ctypes.c_int64)]


class lmc_copy_batch(ctypes.Structure):
    _fields_ = [("num_kv_groups", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("pairs", ctypes.POINTER(ctypes.c_void_p)), ("num_pairs", ctypes.POINTER(ctypes.c_int64)),
                ("host_pairs", ctypes.POINTER(ctypes.c_void_p))]


class lmc_batch(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("num_kv_groups", ctypes.c_int32),
                ("tables", ctypes.POINTER(lmc_block_table)), ("num_object_groups", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("jobs", ctypes.POINTER(ctypes.c_void_p)),
                ("num_jobs", ctypes.POINTER(ctypes.c_int64))]


_P = ctypes.POINTER
_i64 = ctypes.c_int64


def _bind(so: ctypes.CDLL) -> ctypes.CDLL:
    so.lmc_layout_build.argtypes = [_P(lmc_layout_params), _P(ctypes.c_void_p)]
    so.lmc_layout_query.argtypes = [ctypes.c_void_p, _P(lmc_layout_info)]
    so.lmc_layout_free.argtypes = [ctypes.c_void_p]
    so.lmc_layout_free.restype = None
    so.lmc_object_bytes.argtypes = [ctypes.c_void_p, _i64, ctypes.c_int32, _P(_i64)]
    so.lmc_negotiate_chunk.argtypes = [_i64, _i64, ctypes.c_int, _P(_i64)]
    so.lmc_check_step_budget.argtypes = [_i64, _i64, ctypes.c_int]
    so.lmc_unified_block_size.argtypes = [_i64, _i64, _i64, _P(_i64)]
    for name in ("lmc_store", "lmc_load"):
        getattr(so, name).argtypes = [ctypes.c_void_p, _i64, ctypes.c_void_p, _P(lmc_batch), ctypes.c_void_p,
                                      _i64, ctypes.c_void_p, ctypes.c_void_p]
    so.lmc_layout_check_backends.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                             _P(ctypes.c_uint32)]
    so.lmc_object_bytes_blocks.argtypes = [ctypes.c_void_p, _i64, ctypes.c_int32, ctypes.c_int32, _P(_i64)]
    for name in ("lmc_store_blocks", "lmc_load_blocks"):
        getattr(so, name).argtypes = [ctypes.c_void_p, _i64, ctypes.c_int32, ctypes.c_void_p, _P(lmc_batch),
                                      ctypes.c_void_p, _i64, ctypes.c_void_p, ctypes.c_void_p]
    so.lmc_copy_blocks.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _P(lmc_copy_batch), ctypes.c_void_p,
                                   ctypes.c_void_p]
    so.lmc_check_disjoint.argtypes = [ctypes.c_void_p, _i64, _P(lmc_batch), _P(lmc_batch), _P(ctypes.c_int32)]
    so.lmc_check_disjoint_blocks.argtypes = [ctypes.c_void_p, _i64, ctypes.c_int32, _P(lmc_batch), _P(lmc_batch),
                                             _P(ctypes.c_int32)]
    for name in ("lmc_store_q8", "lmc_load_q8"):
        getattr(so, name).argtypes = [ctypes.c_void_p, _i64, _i64, ctypes.c_void_p, _P(lmc_batch), ctypes.c_void_p,
                                      _i64, ctypes.c_void_p, ctypes.c_void_p]
    so.lmc_object_bytes_q8.argtypes = [ctypes.c_void_p, _i64, _i64, ctypes.c_int32, _P(_i64)]
    for name in ("lmc_store_blocks_q8", "lmc_load_blocks_q8"):
        getattr(so, name).argtypes = [ctypes.c_void_p, _i64, ctypes.c_int32, _i64, ctypes.c_void_p,
                                      _P(lmc_batch), ctypes.c_void_p, _i64, ctypes.c_void_p, ctypes.c_void_p]
    so.lmc_object_bytes_blocks_q8.argtypes = [ctypes.c_void_p, _i64, ctypes.c_int32, _i64, ctypes.c_int32, _P(_i64)]
    so.lmc_selftest_wait.argtypes = [ctypes.c_void_p, _i64, ctypes.c_void_p]
    so.lmc_selftest_row_scale.argtypes = [ctypes.c_void_p] * 4 + [_i64, ctypes.c_void_p]
    so.lmc_strerror.argtypes = [ctypes.c_int]
    so.lmc_strerror.restype = ctypes.c_char_p
    return so


def _use_library(path: str) -> None:
    """Binds the package to another build of liblmc (e.g. one compiled with
    other tile constants). Layouts built before the switch must not be used
    after it."""
    global _lib
    _lib = _bind(ctypes.CDLL(path))


_use_library(LIB_PATH)


def lmc_strerror(code: int) -> str:
    return _lib.lmc_strerror(int(code)).decode()


def _check(rc: int, what: str):
    if rc != LMC_OK:
        raise LmcError(rc, what)


# ----------------------------------------------------------------------------
# Host rules
# ----------------------------------------------------------------------------

def lmc_negotiate_chunk(requested: int, block_size: int, strict: bool = False) -> int:
    out = _i64(0)
    _check(_lib.lmc_negotiate_chunk(int(requested), int(block_size), int(bool(strict)), ctypes.byref(out)),
           f"lmc_negotiate_chunk({requested}, {block_size}, strict={strict})")
    return out.value


def lmc_check_step_budget(block_size: int, max_batched: int, separate_object_groups: bool) -> int:
    """Returns the library's code (LMC_OK when the budget is allowed)."""
    return _lib.lmc_check_step_budget(int(block_size), int(max_batched), int(bool(separate_object_groups)))


def lmc_unified_block_size(attn_token_bytes: int, state_page_bytes: int, align: int = 16) -> int:
    out = _i64(0)
    _check(_lib.lmc_unified_block_size(int(attn_token_bytes), int(state_page_bytes), int(align), ctypes.byref(out)),
           "lmc_unified_block_size")
    return out.value


# ----------------------------------------------------------------------------
# Layout
# ----------------------------------------------------------------------------

class Layout:
    """An immutable pool layout built by ``lmc_layout_build`` (freed on GC)."""

    def __init__(self, handle: int):
        self._h = ctypes.c_void_p(handle)
        self._so = _lib  # the build that allocated the handle also frees it
        info = lmc_layout_info()
        _check(_lib.lmc_layout_query(self._h, ctypes.byref(info)), "lmc_layout_query")
        n, g, o = info.num_layers, info.num_kv_groups, info.num_object_groups
        self.num_layers = n
        self.num_kv_groups = g
        self.num_object_groups = o
        self.num_slabs = info.num_slabs
        self.block_size = self.N = info.block_size
        self.page_size = info.page_size
        self.block_stride = info.block_stride
        self.num_blocks = info.num_blocks
        self.pool_bytes = info.pool_bytes
        d = [info.layers[i] for i in range(n)]
        self.kinds = [LMC_LAYER_NAME[x.kind] for x in d]
        self.kv_group = [x.kv_group for x in d]
        self.slot = [x.slot for x in d]
        self.object_group = [x.object_group for x in d]
        self.real_bytes = [x.real_bytes for x in d]
        self.page_bytes = [x.page_bytes for x in d]
        self.base = [x.base for x in d]
        self.stride = [x.stride for x in d]
        self.kv_group_kind = [LMC_LAYER_NAME[info.kv_group_kind[k]] for k in range(g)]
        self.kv_group_size = [info.kv_group_size[k] for k in range(g)]
        self.object_group_kind = [LMC_LAYER_NAME[info.object_group_kind[k]] for k in range(o)]

    @property
    def handle(self):
        return self._h

    def object_bytes(self, chunk: int, object_group: int) -> int:
        return lmc_object_bytes(self, chunk, object_group)

    def check_backends(self, attn_indexes_by_stride: bool, state_pages_strided_ok: bool) -> int:
        return lmc_layout_check_backends(self, attn_indexes_by_stride, state_pages_strided_ok)

    def object_bytes_q8(self, chunk: int, row_elems: int, object_group: int) -> int:
        return lmc_object_bytes_q8(self, chunk, row_elems, object_group)

    def object_bytes_blocks(self, blocks_per_object: int, kda_every: bool, object_group: int) -> int:
        return lmc_object_bytes_blocks(self, blocks_per_object,
                                       LMC_KDA_EVERY_BLOCK if kda_every else LMC_KDA_LAST_BLOCK, object_group)

    def object_bytes_blocks_q8(self, blocks_per_object: int, kda_every: bool, row_elems: int,
                               object_group: int) -> int:
        return lmc_object_bytes_blocks_q8(self, blocks_per_object,
                                          LMC_KDA_EVERY_BLOCK if kda_every else LMC_KDA_LAST_BLOCK, row_elems,
                                          object_group)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._so.lmc_layout_free(h)
            self._h = None


def lmc_layout_build(layers, block_size: int, packed: bool, mem_bytes: int, split_groups: bool = True,
                     separate_object_groups: bool = True) -> Layout:
    """`layers`: model-order list of dicts {"kind", "token_bytes", "conv_bytes", "rec_bytes", "window"}."""
    n = len(layers)
    arr = (lmc_layer_spec * max(n, 1))()
    for i, l in enumerate(layers):
        arr[i] = lmc_layer_spec(LMC_LAYER[l["kind"]], int(l.get("window", 0)), int(l.get("token_bytes", 0)),
                                int(l.get("conv_bytes", 0)), int(l.get("rec_bytes", 0)))
    p = lmc_layout_params(n, 1 if packed else 0, 0 if split_groups else 1, int(bool(separate_object_groups)),
                          int(block_size), int(mem_bytes), arr)
    h = ctypes.c_void_p()
    _check(_lib.lmc_layout_build(ctypes.byref(p), ctypes.byref(h)), "lmc_layout_build")
    return Layout(h.value)


def lmc_layout_check_backends(layout: Layout, attn_indexes_by_stride: bool, state_pages_strided_ok: bool) -> int:
    """LMC_BK_* bits of the eligibility rules the layout breaks (0: readable)."""
    out = ctypes.c_uint32(0)
    _check(_lib.lmc_layout_check_backends(layout.handle, int(bool(attn_indexes_by_stride)),
                                          int(bool(state_pages_strided_ok)), ctypes.byref(out)),
           "lmc_layout_check_backends")
    return out.value


def lmc_object_bytes(layout: Layout, chunk: int, object_group: int) -> int:
    out = _i64(0)
    _check(_lib.lmc_object_bytes(layout.handle, int(chunk), int(object_group), ctypes.byref(out)),
           "lmc_object_bytes")
    return out.value


def lmc_object_bytes_blocks(layout: Layout, blocks_per_object: int, kda_mode: int, object_group: int) -> int:
    out = _i64(0)
    _check(_lib.lmc_object_bytes_blocks(layout.handle, int(blocks_per_object), int(kda_mode), int(object_group),
                                        ctypes.byref(out)), "lmc_object_bytes_blocks")
    return out.value


# ----------------------------------------------------------------------------
# Store / load
# ----------------------------------------------------------------------------

def jobs_to_device(jobs: np.ndarray, device):
    """Uploads a JOB_DTYPE numpy array as a uint8 device tensor of 16-byte records."""
    import torch
    a = np.ascontiguousarray(jobs, dtype=JOB_DTYPE)
    return torch.from_numpy(a.view(np.uint8).copy()).to(device)


def _batch(layout: Layout, tables, jobs):
    g = layout.num_kv_groups
    if len(tables) != g:
        raise LmcError(LMC_ERR_INVALID_ARG, f"{g} block tables expected, got {len(tables)}")
    nreq = int(tables[0].shape[0]) if g else 0
    tarr = (lmc_block_table * max(g, 1))()
    for k, t in enumerate(tables):
        _visible("block table", t)
        if t.dim() != 2 or t.element_size() != 4 or t.stride(1) != 1 or int(t.shape[0]) != nreq:
            raise LmcError(LMC_ERR_INVALID_ARG, "block tables must be int32 [num_requests, cols] with unit column stride")
        tarr[k] = lmc_block_table(t.data_ptr(), int(t.stride(0)), int(t.shape[1]))
    o = layout.num_object_groups
    if len(jobs) != o:
        raise LmcError(LMC_ERR_INVALID_ARG, f"{o} job arrays expected, got {len(jobs)}")
    jarr = (ctypes.c_void_p * max(o, 1))()
    narr = (_i64 * max(o, 1))()
    for q, j in enumerate(jobs):
        _visible("job array", j)
        nbytes = j.numel() * j.element_size()
        if nbytes % 16 or not j.is_contiguous():
            raise LmcError(LMC_ERR_INVALID_ARG, "job arrays hold contiguous 16-byte lmc_job records")
        jarr[q] = j.data_ptr() if nbytes else None
        narr[q] = nbytes // 16
    b = lmc_batch(nreq, g, tarr, o, 0, jarr, narr)
    return b, (tarr, jarr, narr)


def _stream_ptr(stream, *buffers):
    """The stream's handle. When the call runs on a stream other than the
    current one, every device tensor among `buffers` (nested lists
    included) is marked as used by that stream, so that torch's caching
    allocator does not hand its memory to a later allocation before the
    call's kernels have read or written it."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    elif stream != torch.cuda.current_stream(stream.device):
        todo = list(buffers)
        while todo:
            t = todo.pop()
            if isinstance(t, (list, tuple)):
                todo.extend(t)
            elif isinstance(t, torch.Tensor) and t.is_cuda:
                t.record_stream(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _visible(name: str, t) -> None:
    """Refuses memory the kernels could not address: every buffer handed to a
    launch must be a CUDA tensor or pinned (page-locked) host memory."""
    if not (t.is_cuda or t.is_pinned()):
        raise LmcError(LMC_ERR_INVALID_ARG, f"{name} must be a CUDA tensor or pinned host memory")


def _check_launch(layout: Layout, pool, arena, status):
    for name, t in (("pool", pool), ("arena", arena), ("status", status)):
        if t is not None:
            _visible(name, t)
    if pool.numel() * pool.element_size() < layout.pool_bytes:
        raise LmcError(LMC_ERR_INVALID_ARG, f"pool holds {pool.numel() * pool.element_size()} bytes, "
                                            f"the layout addresses {layout.pool_bytes}")


def lmc_store(layout: Layout, chunk: int, pool, tables, jobs, arena, status, stream=None) -> None:
    """Gathers the jobs' objects from `pool` into `arena` (device tensors) on
    `stream` (default: torch's current stream). Device errors are OR-ed into
    the 4-byte `status` tensor."""
    _check_launch(layout, pool, arena, status)
    b, keep = _batch(layout, tables, jobs)
    strm = _stream_ptr(stream, pool, tables, jobs, arena, status)
    _check(_lib.lmc_store(layout.handle, int(chunk), pool.data_ptr(), ctypes.byref(b), arena.data_ptr(),
                          arena.numel() * arena.element_size(), status.data_ptr(), strm),
           "lmc_store")


def lmc_load(layout: Layout, chunk: int, pool, tables, jobs, arena, status, stream=None) -> None:
    """Scatters the jobs' objects from `arena` into `pool` (device tensors)."""
    _check_launch(layout, pool, arena, status)
    b, keep = _batch(layout, tables, jobs)
    strm = _stream_ptr(stream, pool, tables, jobs, arena, status)
    _check(_lib.lmc_load(layout.handle, int(chunk), pool.data_ptr(), ctypes.byref(b), arena.data_ptr(),
                         arena.numel() * arena.element_size(), status.data_ptr(), strm),
           "lmc_load")


def lmc_store_blocks(layout: Layout, blocks_per_object: int, kda_mode: int, pool, tables, jobs, arena, status,
                     stream=None) -> None:
    """Block-granular store: each job's `chunk` field is its first block position."""
    _check_launch(layout, pool, arena, status)
    b, keep = _batch(layout, tables, jobs)
    strm = _stream_ptr(stream, pool, tables, jobs, arena, status)
    _check(_lib.lmc_store_blocks(layout.handle, int(blocks_per_object), int(kda_mode), pool.data_ptr(),
                                 ctypes.byref(b), arena.data_ptr(), arena.numel() * arena.element_size(),
                                 status.data_ptr(), strm), "lmc_store_blocks")


def lmc_load_blocks(layout: Layout, blocks_per_object: int, kda_mode: int, pool, tables, jobs, arena, status,
                    stream=None) -> None:
    _check_launch(layout, pool, arena, status)
    b, keep = _batch(layout, tables, jobs)
    strm = _stream_ptr(stream, pool, tables, jobs, arena, status)
    _check(_lib.lmc_load_blocks(layout.handle, int(blocks_per_object), int(kda_mode), pool.data_ptr(),
                                ctypes.byref(b), arena.data_ptr(), arena.numel() * arena.element_size(),
                                status.data_ptr(), strm), "lmc_load_blocks")


def lmc_object_bytes_q8(layout: Layout, chunk: int, row_elems: int, object_group: int) -> int:
    out = _i64(0)
    _check(_lib.lmc_object_bytes_q8(layout.handle, int(chunk), int(row_elems), int(object_group),
                                    ctypes.byref(out)), "lmc_object_bytes_q8")
    return out.value


def lmc_store_q8(layout: Layout, chunk: int, row_elems: int, pool, tables, jobs, arena, status,
                 stream=None) -> None:
    """Chunk store with KDA snapshots as INT8 records (rows of `row_elems`)."""
    _check_launch(layout, pool, arena, status)
    b, keep = _batch(layout, tables, jobs)
    strm = _stream_ptr(stream, pool, tables, jobs, arena, status)
    _check(_lib.lmc_store_q8(layout.handle, int(chunk), int(row_elems), pool.data_ptr(), ctypes.byref(b),
                             arena.data_ptr(), arena.numel() * arena.element_size(), status.data_ptr(), strm),
           "lmc_store_q8")


def lmc_load_q8(layout: Layout, chunk: int, row_elems: int, pool, tables, jobs, arena, status,
                stream=None) -> None:
    _check_launch(layout, pool, arena, status)
    b, keep = _batch(layout, tables, jobs)
    strm = _stream_ptr(stream, pool, tables, jobs, arena, status)
    _check(_lib.lmc_load_q8(layout.handle, int(chunk), int(row_elems), pool.data_ptr(), ctypes.byref(b),
                            arena.data_ptr(), arena.numel() * arena.element_size(), status.data_ptr(), strm),
           "lmc_load_q8")


def lmc_object_bytes_blocks_q8(layout: Layout, blocks_per_object: int, kda_mode: int, row_elems: int,
                               object_group: int) -> int:
    out = _i64(0)
    _check(_lib.lmc_object_bytes_blocks_q8(layout.handle, int(blocks_per_object), int(kda_mode), int(row_elems),
                                           int(object_group), ctypes.byref(out)), "lmc_object_bytes_blocks_q8")
    return out.value


def lmc_store_blocks_q8(layout: Layout, blocks_per_object: int, kda_mode: int, row_elems: int, pool, tables, jobs,
                        arena, status, stream=None) -> None:
    """Block-granular store with the stored KDA snapshots as INT8 records."""
    _check_launch(layout, pool, arena, status)
    b, keep = _batch(layout, tables, jobs)
    strm = _stream_ptr(stream, pool, tables, jobs, arena, status)
    _check(_lib.lmc_store_blocks_q8(layout.handle, int(blocks_per_object), int(kda_mode), int(row_elems),
                                    pool.data_ptr(), ctypes.byref(b), arena.data_ptr(),
                                    arena.numel() * arena.element_size(), status.data_ptr(), strm),
           "lmc_store_blocks_q8")


def lmc_load_blocks_q8(layout: Layout, blocks_per_object: int, kda_mode: int, row_elems: int, pool, tables, jobs,
                       arena, status, stream=None) -> None:
    _check_launch(layout, pool, arena, status)
    b, keep = _batch(layout, tables, jobs)
    strm = _stream_ptr(stream, pool, tables, jobs, arena, status)
    _check(_lib.lmc_load_blocks_q8(layout.handle, int(blocks_per_object), int(kda_mode), int(row_elems),
                                   pool.data_ptr(), ctypes.byref(b), arena.data_ptr(),
                                   arena.numel() * arena.element_size(), status.data_ptr(), strm),
           "lmc_load_blocks_q8")


def lmc_selftest_wait(status, rounds: int, stream=None) -> None:
    """Runs the bounded-wait self-test: LMC_ST_TIMEOUT lands in `status`."""
    strm = _stream_ptr(stream, status)
    _check(_lib.lmc_selftest_wait(status.data_ptr(), int(rounds), strm), "lmc_selftest_wait")


def lmc_selftest_row_scale(amax, scale, inv, ieee, stream=None) -> None:
    """The codec's row scale and inverse for each value of the float32
    device tensor `amax`, with CUDA's IEEE quotient amax / 127 beside them."""
    n = amax.numel()
    for t in (scale, inv, ieee):
        if t.numel() != n:
            raise ValueError("lmc_selftest_row_scale: output sizes differ from amax")
    strm = _stream_ptr(stream, amax, scale, inv, ieee)
    _check(_lib.lmc_selftest_row_scale(amax.data_ptr(), scale.data_ptr(), inv.data_ptr(), ieee.data_ptr(), n, strm),
           "lmc_selftest_row_scale")


def pairs_to_device(pairs: np.ndarray, device):
    """Uploads a PAIR_DTYPE numpy array as a uint8 device tensor of 8-byte records."""
    import torch
    a = np.ascontiguousarray(pairs, dtype=PAIR_DTYPE)
    return torch.from_numpy(a.view(np.uint8).copy()).to(device)


def lmc_copy_blocks(layout: Layout, pool, pairs, host_pairs, status, stream=None) -> None:
    """In-pool copies: `pairs[g]` (device tensor of 8-byte lmc_block_pair
    records) lists (src, dst) blocks of KV group g; `host_pairs[g]` is the
    same list as a PAIR_DTYPE numpy array, on which the library checks that
    the copies do not race (LmcError LMC_ERR_OVERLAP otherwise)."""
    _check_launch(layout, pool, None, status)
    g = layout.num_kv_groups
    if len(pairs) != g or len(host_pairs) != g:
        raise LmcError(LMC_ERR_INVALID_ARG, f"{g} pair arrays expected, got {len(pairs)} and {len(host_pairs)}")
    parr = (ctypes.c_void_p * max(g, 1))()
    harr = (ctypes.c_void_p * max(g, 1))()
    narr = (_i64 * max(g, 1))()
    keep = []
    for k, (p, h) in enumerate(zip(pairs, host_pairs)):
        _visible("pair array", p)
        nbytes = p.numel() * p.element_size()
        if nbytes % 8 or not p.is_contiguous():
            raise LmcError(LMC_ERR_INVALID_ARG, "pair arrays hold contiguous 8-byte lmc_block_pair records")
        h = np.ascontiguousarray(h, dtype=PAIR_DTYPE)
        if h.nbytes != nbytes:
            raise LmcError(LMC_ERR_INVALID_ARG, "host and device pair arrays differ in length")
        keep.append(h)
        parr[k] = p.data_ptr() if nbytes else None
        harr[k] = h.ctypes.data if nbytes else None
        narr[k] = nbytes // 8
    b = lmc_copy_batch(g, 0, parr, narr, harr)
    strm = _stream_ptr(stream, pool, pairs, status)
    _check(_lib.lmc_copy_blocks(layout.handle, pool.data_ptr(), ctypes.byref(b), status.data_ptr(), strm),
           "lmc_copy_blocks")


def _host_batch(layout: Layout, tables, jobs):
    """An lmc_batch over HOST numpy arrays (int32 block tables, JOB_DTYPE jobs)."""
    g = layout.num_kv_groups
    if len(tables) != g or len(jobs) != layout.num_object_groups:
        raise LmcError(LMC_ERR_INVALID_ARG, "one block table per KV group and one job array per object group")
    keep = []
    nreq = int(tables[0].shape[0]) if g else 0
    tarr = (lmc_block_table * max(g, 1))()
    for k, t in enumerate(tables):
        t = np.ascontiguousarray(t, dtype=np.int32)
        if t.ndim != 2 or t.shape[0] != nreq:
            raise LmcError(LMC_ERR_INVALID_ARG, "block tables must be int32 [num_requests, cols]")
        keep.append(t)
        tarr[k] = lmc_block_table(t.ctypes.data, int(t.shape[1]), int(t.shape[1]))
    o = layout.num_object_groups
    jarr = (ctypes.c_void_p * max(o, 1))()
    narr = (_i64 * max(o, 1))()
    for q, j in enumerate(jobs):
        j = np.ascontiguousarray(j, dtype=JOB_DTYPE)
        keep.append(j)
        jarr[q] = j.ctypes.data if j.size else None
        narr[q] = j.size
    return lmc_batch(nreq, g, tarr, o, 0, jarr, narr), (keep, tarr, jarr, narr)


def lmc_check_disjoint(layout: Layout, chunk: int, tables_a, jobs_a, tables_b, jobs_b) -> int:
    """Host check for two chunk batches run at the same time on one pool
    (numpy block tables and JOB_DTYPE jobs): -1 when the blocks their
    objects touch are disjoint, else the smallest block both touch."""
    a, keep_a = _host_batch(layout, tables_a, jobs_a)
    b, keep_b = _host_batch(layout, tables_b, jobs_b)
    out = ctypes.c_int32(0)
    rc = _lib.lmc_check_disjoint(layout.handle, int(chunk), ctypes.byref(a), ctypes.byref(b), ctypes.byref(out))
    if rc == LMC_ERR_OVERLAP:
        return out.value
    _check(rc, "lmc_check_disjoint")
    return -1


def lmc_check_disjoint_blocks(layout: Layout, blocks_per_object: int, kda_mode: int, tables_a, jobs_a, tables_b,
                              jobs_b) -> int:
    """lmc_check_disjoint for block-granular batches (jobs name their first
    block position): -1 when disjoint, else the smallest shared block."""
    a, keep_a = _host_batch(layout, tables_a, jobs_a)
    b, keep_b = _host_batch(layout, tables_b, jobs_b)
    out = ctypes.c_int32(0)
    rc = _lib.lmc_check_disjoint_blocks(layout.handle, int(blocks_per_object), int(kda_mode), ctypes.byref(a),
                                        ctypes.byref(b), ctypes.byref(out))
    if rc == LMC_ERR_OVERLAP:
        return out.value
    _check(rc, "lmc_check_disjoint_blocks")
    return -1


__all__ = [n for n in dir() if n.startswith(("lmc_", "LMC_"))] + ["Layout", "LmcError", "JOB_DTYPE",
                                                                  "jobs_to_device",
                                                                  "PAIR_DTYPE", "pairs_to_device"]

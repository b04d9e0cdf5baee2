"""Per-token numpy brute force of the cache paging (test infrastructure only).

A second, independent restatement used to check ``oracle.c`` on tiny pools.
It shares nothing with the C oracle: it derives its own layout by following
the steps the vLLM blog describes ("How vLLM manages the KV cache of hybrid
models", §2.2 grouping, §3.1 path A shared tensors, §3.2 path B packed offsets,
§4 the int8 buffer and its per-layer views), builds numpy views of the pool
exactly as those sections describe, and moves bytes one token at a time.

Only valid inputs are handled (no error bits): it is a cross-check of the
arithmetic, not of the error paths.
"""
from __future__ import annotations

import math
from collections import OrderedDict

import numpy as np
from numpy.lib.stride_tricks import as_strided


def _spec_key(l):
    return (l["kind"], int(l.get("token_bytes", 0)), int(l.get("conv_bytes", 0)),
            int(l.get("rec_bytes", 0)), int(l.get("window", 0)))


def _page_bytes(l, N):
    # KDA: conv_state + recurrent_state, independent of length (§2.1);
    # paged attention: N tokens of token_bytes each (§4.2).
    if l["kind"] == "KDA":
        return int(l["conv_bytes"]) + int(l["rec_bytes"])
    return N * int(l["token_bytes"])


def groups(spec_layers, split_groups=True):
    """KV cache groups as lists of layer indices (§2.2, then the equal split
    that puts K3's 69 KDA layers on 23-layer groups)."""
    same_type = OrderedDict()
    for i, l in enumerate(spec_layers):
        same_type.setdefault(_spec_key(l), []).append(i)
    if not split_groups:
        return [list(v) for v in same_type.values()]
    smallest = min(len(v) for v in same_type.values())
    out = []
    for v in same_type.values():
        parts = math.ceil(len(v) / smallest)
        out += [list(map(int, p)) for p in np.array_split(np.array(v), parts)]
    return out


def object_groups(spec_layers, separate=True):
    """Object groups as lists of layer indices in model order
    ("Hybrid Attention Models", Object-group separation)."""
    if not separate:
        return [list(range(len(spec_layers)))]
    classes = OrderedDict()
    for i, l in enumerate(spec_layers):
        cls = ("SWA", int(l["window"])) if l["kind"] == "SWA" else (l["kind"],)
        classes.setdefault(cls, []).append(i)
    return list(classes.values())


class BruteLayout:
    """Pool geometry plus one numpy view per layer over a pool buffer."""

    def __init__(self, spec_layers, N, packed, mem_bytes, split_groups=True):
        self.spec = spec_layers
        self.N = N
        self.packed = packed
        self.groups = groups(spec_layers, split_groups)
        pages = [_page_bytes(l, N) for l in spec_layers]
        self.pages = pages
        if not packed:
            # Path A: page_size is the largest page; tensor t (size
            # page_size * num_blocks) is shared_by the t-th layer of each group.
            page_size = max(pages)
            S = max(len(g) for g in self.groups)
            num_blocks = mem_bytes // (page_size * S)
            self.tensor_offset = {}
            self.layer_stride = {}
            for t in range(S):
                for g in self.groups:
                    if t < len(g):
                        self.tensor_offset[g[t]] = t * page_size * num_blocks
                        self.layer_stride[g[t]] = page_size
            self.pool_bytes = S * page_size * num_blocks
        else:
            # Path B: per group, byte_offset accumulates each layer's page;
            # block_stride = max over groups; num_blocks = memory // stride.
            block_stride = 0
            self.tensor_offset = {}
            for g in self.groups:
                byte_offset = 0
                for i in g:
                    self.tensor_offset[i] = byte_offset
                    byte_offset += pages[i]
                block_stride = max(block_stride, byte_offset)
            num_blocks = mem_bytes // block_stride
            self.layer_stride = {i: block_stride for i in range(len(spec_layers))}
            self.pool_bytes = num_blocks * block_stride
        self.num_blocks = num_blocks
        self.kv_group_of = {i: k for k, g in enumerate(self.groups) for i in g}

    def view(self, pool: np.ndarray, i: int) -> np.ndarray:
        """Layer i's cache as vLLM's backends see it: (num_blocks, N, token_bytes)
        for paged attention, (num_blocks, page_bytes) for KDA."""
        l = self.spec[i]
        off = self.tensor_offset[i]
        st = self.layer_stride[i]
        if l["kind"] == "KDA":
            return as_strided(pool[off:], shape=(self.num_blocks, self.pages[i]), strides=(st, 1),
                              writeable=pool.flags.writeable)
        tb = int(l["token_bytes"])
        return as_strided(pool[off:], shape=(self.num_blocks, self.N, tb), strides=(st, tb, 1),
                          writeable=pool.flags.writeable)


def _object_pieces(BL: BruteLayout, og_layers, tables, r, first_tok, ntok, kda_every=False):
    """Yields (layer, view index tuple) in object order for the object that
    covers tokens [first_tok, first_tok + ntok): one token at a time for
    paged layers; for KDA layers the snapshot taken after the object's last
    token, or, with kda_every, the snapshot after each of its blocks."""
    N = BL.N
    for i in og_layers:
        row = tables[BL.kv_group_of[i]][r]
        if BL.spec[i]["kind"] == "KDA":
            ends = range(first_tok + N, first_tok + ntok + 1, N) if kda_every else [first_tok + ntok]
            for end_tok in ends:
                # the state after `end_tok` tokens lives in the block ending there
                yield i, (int(row[end_tok // N - 1]),)
        else:
            for t in range(first_tok, first_tok + ntok):
                yield i, (int(row[t // N]), t % N)


def _span(BL, job, C, nb):
    """Token range of a job: chunk jobs cover chunk * C .. + C; block jobs
    (nb > 0) cover their first block's tokens onward for nb blocks."""
    if nb:
        return int(job["chunk"]) * BL.N, nb * BL.N
    return int(job["chunk"]) * C, C


def store(BL: BruteLayout, C, pool, tables, jobs, arena, separate=True, nb=0, kda_every=False):
    ogs = object_groups(BL.spec, separate)
    for og, layers in enumerate(ogs):
        for job in jobs[og]:
            first, n = _span(BL, job, C, nb)
            parts = [BL.view(pool, i)[idx].reshape(-1)
                     for i, idx in _object_pieces(BL, layers, tables, int(job["request"]), first, n, kda_every)]
            blob = np.concatenate(parts)
            off = int(job["offset"])
            arena[off:off + blob.size] = blob


def load(BL: BruteLayout, C, pool, tables, jobs, arena, separate=True, nb=0, kda_every=False):
    ogs = object_groups(BL.spec, separate)
    for og, layers in enumerate(ogs):
        for job in jobs[og]:
            first, n = _span(BL, job, C, nb)
            cur = int(job["offset"])
            for i, idx in _object_pieces(BL, layers, tables, int(job["request"]), first, n, kda_every):
                v = BL.view(pool, i)
                k = v[idx].size
                v[idx] = arena[cur:cur + k].reshape(v[idx].shape)
                cur += k


def copy_blocks(BL: BruteLayout, pool, pairs):
    """pairs[g]: (src, dst) block pairs of KV group g; every layer's view row
    dst takes row src."""
    for g, P in enumerate(pairs):
        for p in P:
            for i in BL.groups[g]:
                v = BL.view(pool, i)
                v[int(p["dst_block"])] = v[int(p["src_block"])].copy()

// layout.cpp -- host-side pool layout, chunk negotiation and the scheduler
// budget rule of liblmc.
//
// Pages followed (title, section):
//   "How vLLM manages the KV cache of hybrid models: Kimi Linear / Kimi K3",
//     §2.1 (KDA conv/recurrent state shapes), §2.2 (KV cache groups are
//     keyed by equal specs), §3.1 (path A: one page size, shared tensors,
//     offset = block_id * page_size), §3.2 (path B: per-group cumulative
//     offsets, block_stride = max group total, num_blocks = mem // stride).
//   "When Prefix Cache Meets KDA" (Mooncake post), "Flat KV": K3's 69 KDA
//     layers form three groups of 23 which with the full-attention group
//     occupy 24 slabs.
//   "Hybrid Attention Models" (LMCache docs), "Object-group separation".
//   "Kimi K3" (LMCache recipe), chunk-size negotiation; "Kimi-Linear"
//     (LMCache recipe), strict multiple rule and the [N, 2N) budget.
#include <algorithm>
#include <cstring>
#include <map>
#include <new>
#include <tuple>

#include "lmc_internal.h"

namespace {

using SpecKey = std::tuple<int32_t, int64_t, int64_t, int64_t, int32_t>;

// Layers form one KV cache group only if their specs are equal field by
// field (§2.2: same_type_layers keyed by the spec value).
SpecKey key_of(const lmc_layer_spec &s) {
    return SpecKey(s.kind, s.token_bytes, s.conv_bytes, s.rec_bytes, s.window);
}

// Object-group class ("Hybrid Attention Models", Object-group separation):
// full attention is one cross-chunk window, KDA (mamba-like) another, each
// sliding-window size another.
std::pair<int32_t, int32_t> window_class(const lmc_layer_spec &s) {
    return {s.kind, s.kind == LMC_LAYER_SWA ? s.window : 0};
}

int validate_spec(const lmc_layer_spec &s, int64_t N, int64_t *real) {
    switch (s.kind) {
    case LMC_LAYER_KDA:
        if (s.conv_bytes < 0 || s.rec_bytes < 0)
            return LMC_ERR_INVALID_ARG;
        if (!lmc::add_ok(s.conv_bytes, s.rec_bytes, real))
            return LMC_ERR_OVERFLOW;
        return *real > 0 ? LMC_OK : LMC_ERR_INVALID_ARG;
    case LMC_LAYER_SWA:
        if (s.window <= 0)
            return LMC_ERR_INVALID_ARG;
        [[fallthrough]];
    case LMC_LAYER_MLA:
        if (s.token_bytes <= 0)
            return LMC_ERR_INVALID_ARG;
        return lmc::mul_ok(N, s.token_bytes, real) ? LMC_OK : LMC_ERR_OVERFLOW;
    default:
        return LMC_ERR_INVALID_ARG;
    }
}

}  // namespace

extern "C" int lmc_layout_build(const lmc_layout_params *p, lmc_layout **out) {
    if (p == nullptr || out == nullptr || p->layers == nullptr)
        return LMC_ERR_INVALID_ARG;
    const int n = p->num_layers;
    if (n <= 0 || n > LMC_MAX_LAYERS || p->block_size <= 0 || p->mem_bytes < 0)
        return LMC_ERR_INVALID_ARG;
    if (p->mode != LMC_LAYOUT_PADDED && p->mode != LMC_LAYOUT_PACKED)
        return LMC_ERR_INVALID_ARG;
    if (p->grouping != LMC_GROUP_SPLIT && p->grouping != LMC_GROUP_BY_SPEC)
        return LMC_ERR_INVALID_ARG;

    lmc_layout *L = new (std::nothrow) lmc_layout();
    if (L == nullptr)
        return LMC_ERR_INVALID_ARG;
    L->block_size = p->block_size;
    L->mode = p->mode;
    L->specs.assign(p->layers, p->layers + n);
    L->desc.assign(n, lmc_layer_desc{});

    auto fail = [&](int rc) {
        delete L;
        return rc;
    };

    for (int i = 0; i < n; i++) {
        int rc = validate_spec(L->specs[i], p->block_size, &L->desc[i].real_bytes);
        if (rc != LMC_OK)
            return fail(rc);
        L->desc[i].kind = L->specs[i].kind;
    }

    // KV cache groups: bucket by spec (first appearance order), then split
    // each bucket into consecutive near-equal runs.
    std::vector<SpecKey> spec_order;
    std::map<SpecKey, std::vector<int>> bucket;
    for (int i = 0; i < n; i++) {
        SpecKey k = key_of(L->specs[i]);
        auto it = bucket.find(k);
        if (it == bucket.end()) {
            spec_order.push_back(k);
            bucket[k] = {i};
        } else {
            it->second.push_back(i);
        }
    }
    size_t smallest = SIZE_MAX;
    for (auto &k : spec_order)
        smallest = std::min(smallest, bucket[k].size());
    int32_t group = 0;
    for (auto &k : spec_order) {
        const std::vector<int> &members = bucket[k];
        const size_t count = members.size();
        const size_t runs = p->grouping == LMC_GROUP_SPLIT ? (count + smallest - 1) / smallest : 1;
        size_t next = 0;
        for (size_t r = 0; r < runs; r++) {
            // the first count % runs runs take one extra layer
            const size_t len = count / runs + (r < count % runs ? 1 : 0);
            for (size_t t = 0; t < len; t++) {
                lmc_layer_desc &d = L->desc[members[next + t]];
                d.kv_group = group;
                d.slot = (int32_t)t;
            }
            L->kv_group_kind.push_back(std::get<0>(k));
            L->kv_group_size.push_back((int32_t)len);
            L->num_slabs = std::max<int32_t>(L->num_slabs, (int32_t)len);
            next += len;
            group++;
        }
    }

    // Object groups.
    std::vector<std::pair<int32_t, int32_t>> classes;
    for (int i = 0; i < n; i++) {
        int32_t og = 0;
        if (p->separate_object_groups) {
            auto c = window_class(L->specs[i]);
            auto it = std::find(classes.begin(), classes.end(), c);
            og = (int32_t)(it - classes.begin());
            if (it == classes.end())
                classes.push_back(c);
        }
        L->desc[i].object_group = og;
        if ((size_t)og >= L->object_group_layers.size()) {
            L->object_group_layers.resize(og + 1);
            L->object_group_kind.push_back(L->specs[i].kind);
        }
        L->object_group_layers[og].push_back(i);
    }

    if (p->mode == LMC_LAYOUT_PADDED) {
        // Path A: every page padded to the largest real page.
        int64_t page = 0;
        for (auto &d : L->desc)
            page = std::max(page, d.real_bytes);
        int64_t per_block, slab_bytes;
        if (!lmc::mul_ok(page, L->num_slabs, &per_block))
            return fail(LMC_ERR_OVERFLOW);
        const int64_t nb = p->mem_bytes / per_block;
        if (nb <= 0)
            return fail(LMC_ERR_NO_MEMORY);
        if (!lmc::mul_ok(page, nb, &slab_bytes))
            return fail(LMC_ERR_OVERFLOW);
        L->page_size = page;
        L->block_stride = page;
        L->num_blocks = nb;
        L->pool_bytes = slab_bytes * L->num_slabs;
        for (auto &d : L->desc) {
            d.page_bytes = page;
            d.stride = page;
            d.base = (int64_t)d.slot * slab_bytes;
        }
    } else {
        // Path B: cumulative offsets inside each group (slot order = model
        // order), block stride = the largest group total.
        std::vector<int64_t> total(L->kv_group_kind.size(), 0);
        for (auto &d : L->desc) {
            d.base = total[d.kv_group];
            d.page_bytes = d.real_bytes;
            if (!lmc::add_ok(total[d.kv_group], d.real_bytes, &total[d.kv_group]))
                return fail(LMC_ERR_OVERFLOW);
        }
        const int64_t stride = *std::max_element(total.begin(), total.end());
        const int64_t nb = p->mem_bytes / stride;
        if (nb <= 0)
            return fail(LMC_ERR_NO_MEMORY);
        L->page_size = 0;
        L->block_stride = stride;
        L->num_blocks = nb;
        L->pool_bytes = nb * stride;  // <= mem_bytes, cannot overflow
        for (auto &d : L->desc)
            d.stride = stride;
    }
    *out = L;
    return LMC_OK;
}

extern "C" int lmc_layout_query(const lmc_layout *L, lmc_layout_info *out) {
    if (L == nullptr || out == nullptr)
        return LMC_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof(*out));
    out->num_layers = (int32_t)L->desc.size();
    out->num_kv_groups = (int32_t)L->kv_group_kind.size();
    out->num_object_groups = (int32_t)L->object_group_layers.size();
    out->num_slabs = L->num_slabs;
    out->block_size = L->block_size;
    out->page_size = L->page_size;
    out->block_stride = L->block_stride;
    out->num_blocks = L->num_blocks;
    out->pool_bytes = L->pool_bytes;
    out->layers = L->desc.data();
    out->kv_group_kind = L->kv_group_kind.data();
    out->kv_group_size = L->kv_group_size.data();
    out->object_group_kind = L->object_group_kind.data();
    return LMC_OK;
}

extern "C" void lmc_layout_free(lmc_layout *L) { delete L; }

extern "C" int lmc_layout_check_backends(const lmc_layout *L, int attn_indexes_by_stride,
                                         int state_pages_strided_ok, uint32_t *out_bits) {
    if (L == nullptr || out_bits == nullptr)
        return LMC_ERR_INVALID_ARG;
    uint32_t bits = 0;
    for (const lmc_layer_desc &d : L->desc) {
        const bool attention = d.kind != LMC_LAYER_KDA;
        if (L->mode == LMC_LAYOUT_PADDED) {
            // vLLM pads a smaller page up to the unified one; for attention
            // that is only legal when the backend strides by block
            if (attention && d.page_bytes > d.real_bytes && !attn_indexes_by_stride)
                bits |= LMC_BK_PADDED_ATTENTION;
        } else if (attention) {
            if (!attn_indexes_by_stride)
                bits |= LMC_BK_PACKED_ATTENTION;
        } else if (!state_pages_strided_ok) {
            bits |= LMC_BK_PACKED_STATE;
        }
    }
    *out_bits = bits;
    return LMC_OK;
}

extern "C" int lmc_object_bytes(const lmc_layout *L, int64_t chunk, int32_t og, int64_t *out) {
    if (L == nullptr || out == nullptr || og < 0 || (size_t)og >= L->object_group_layers.size())
        return LMC_ERR_INVALID_ARG;
    if (chunk <= 0 || chunk % L->block_size != 0)
        return LMC_ERR_NOT_MULTIPLE;
    const int64_t m = chunk / L->block_size;
    int64_t total = 0;
    for (int32_t i : L->object_group_layers[og]) {
        const lmc_layer_desc &d = L->desc[i];
        int64_t part = d.real_bytes;
        if (d.kind != LMC_LAYER_KDA && !lmc::mul_ok(m, d.real_bytes, &part))
            return LMC_ERR_OVERFLOW;
        if (!lmc::add_ok(total, part, &total))
            return LMC_ERR_OVERFLOW;
    }
    *out = total;
    return LMC_OK;
}

extern "C" int lmc_object_bytes_blocks(const lmc_layout *L, int64_t nb, int32_t kda_mode, int32_t og,
                                       int64_t *out) {
    if (L == nullptr || out == nullptr || og < 0 || (size_t)og >= L->object_group_layers.size() || nb <= 0 ||
        (kda_mode != LMC_KDA_LAST_BLOCK && kda_mode != LMC_KDA_EVERY_BLOCK))
        return LMC_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int32_t i : L->object_group_layers[og]) {
        const lmc_layer_desc &d = L->desc[i];
        int64_t part = d.real_bytes;
        const bool one = d.kind == LMC_LAYER_KDA && kda_mode == LMC_KDA_LAST_BLOCK;
        if (!one && !lmc::mul_ok(nb, d.real_bytes, &part))
            return LMC_ERR_OVERFLOW;
        if (!lmc::add_ok(total, part, &total))
            return LMC_ERR_OVERFLOW;
    }
    *out = total;
    return LMC_OK;
}

extern "C" int lmc_negotiate_chunk(int64_t requested, int64_t N, int strict, int64_t *out) {
    if (out == nullptr || N <= 0)
        return LMC_ERR_INVALID_ARG;
    if (strict) {
        if (requested <= 0)
            return LMC_ERR_INVALID_ARG;
        if (requested % N)
            return LMC_ERR_NOT_MULTIPLE;
        *out = requested;
        return LMC_OK;
    }
    if (requested <= N) {
        *out = N;
        return LMC_OK;
    }
    // requested > N > 0: round up without forming requested + N - 1.
    const int64_t q = requested / N + (requested % N != 0);
    int64_t r;
    if (!lmc::mul_ok(q, N, &r))
        return LMC_ERR_OVERFLOW;
    *out = r;
    return LMC_OK;
}

extern "C" int lmc_check_step_budget(int64_t N, int64_t budget, int separate) {
    if (N <= 0 || budget <= 0)
        return LMC_ERR_INVALID_ARG;
    if (budget < N)
        return LMC_ERR_BUDGET;
    // A step of >= 2N tokens spans several blocks and snapshots only its last
    // one; that is allowed only when KDA state has objects of its own.
    if (budget / 2 >= N)  // budget >= 2N without overflow
        return separate ? LMC_OK : LMC_ERR_BUDGET;
    return LMC_OK;
}

extern "C" int lmc_unified_block_size(int64_t attn_token_bytes, int64_t state_page_bytes,
                                      int64_t align, int64_t *out) {
    if (out == nullptr || attn_token_bytes <= 0 || state_page_bytes <= 0 || align <= 0)
        return LMC_ERR_INVALID_ARG;
    // tokens needed so that N * attn_token_bytes >= state_page_bytes ...
    const int64_t tokens = state_page_bytes / attn_token_bytes + (state_page_bytes % attn_token_bytes != 0);
    // ... rounded up to the kernel block alignment.
    const int64_t q = tokens / align + (tokens % align != 0);
    int64_t r;
    if (!lmc::mul_ok(q, align, &r))
        return LMC_ERR_OVERFLOW;
    *out = r;
    return LMC_OK;
}

extern "C" const char *lmc_strerror(int code) {
    switch (code) {
    case LMC_OK: return "LMC_OK: success";
    case LMC_ERR_INVALID_ARG: return "LMC_ERR_INVALID_ARG: invalid argument";
    case LMC_ERR_ALIGN: return "LMC_ERR_ALIGN: misaligned pointer";
    case LMC_ERR_NOT_MULTIPLE: return "LMC_ERR_NOT_MULTIPLE: chunk size is not a positive multiple of the block size";
    case LMC_ERR_NO_MEMORY: return "LMC_ERR_NO_MEMORY: memory holds no whole block of the layout";
    case LMC_ERR_CUDA: return "LMC_ERR_CUDA: a CUDA runtime call failed";
    case LMC_ERR_OVERFLOW: return "LMC_ERR_OVERFLOW: size overflows 64-bit arithmetic";
    case LMC_ERR_BUDGET: return "LMC_ERR_BUDGET: scheduler budget outside [N, 2N) (>= 2N needs separate object groups)";
    case LMC_ERR_OVERLAP: return "LMC_ERR_OVERLAP: copies would race (a block written twice, or written and read)";
    default: return "LMC_ERR_UNKNOWN: unknown status code";
    }
}

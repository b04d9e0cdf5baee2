// checks.cpp -- host-side checks of the preconditions that make concurrent
// copies deterministic: the pairs of one in-pool block copy call, and the two
// batches of a mixed serving step that run at the same time on one pool.
//
// A block id names the same physical block in every KV group: in the padded
// layout the t-th layer of every group shares slab t ("How vLLM manages the
// KV cache of hybrid models", §3.1), and in the packed layout every group's
// pages of block b lie inside [b * block_stride, (b + 1) * block_stride)
// (§3.2). So both checks compare block ids across all KV groups.
#include <algorithm>
#include <cstdint>
#include <iterator>
#include <utility>
#include <vector>

#include "lmc_internal.h"

namespace {

bool valid_block(int64_t b, int64_t num_blocks) { return b >= 0 && b < num_blocks; }

// Blocks whose pages the objects of `b` read (store) or write (load). An
// object covers nb block positions from job.chunk * pos_mul (chunk form:
// pos_mul = nb = C / N; block form: pos_mul = 1): all nb positions of a
// paged layer's block table, and of a KDA layer's either the last one or,
// with kda_every, all nb. Entries the kernels would skip (a request or chunk
// out of range, a position past the table, -1 or an id outside the pool)
// touch nothing. Appends the ids to `out`.
int touched_blocks(const lmc_layout *L, int64_t nb, int64_t pos_mul, bool kda_every, const lmc_batch *b,
                   std::vector<int32_t> &out) {
    const int nkv = (int)L->kv_group_kind.size();
    const int nog = (int)L->object_group_layers.size();
    if (b == nullptr || b->num_requests < 0 || b->num_kv_groups != nkv || b->num_object_groups != nog ||
        (nkv > 0 && b->tables == nullptr) || b->num_jobs == nullptr || b->jobs == nullptr)
        return LMC_ERR_INVALID_ARG;
    for (int k = 0; k < nkv; k++) {
        const lmc_block_table &t = b->tables[k];
        if (t.num_cols < 0 || t.row_stride < t.num_cols || (b->num_requests > 0 && t.num_cols > 0 && t.table == nullptr))
            return LMC_ERR_INVALID_ARG;
    }
    for (int og = 0; og < nog; og++) {
        const int64_t nj = b->num_jobs[og];
        if (nj < 0 || (nj > 0 && b->jobs[og] == nullptr))
            return LMC_ERR_INVALID_ARG;
        // (KV group, KDA?) pairs of the group's layers
        std::vector<std::pair<int32_t, bool>> reads;
        for (int32_t i : L->object_group_layers[og]) {
            const std::pair<int32_t, bool> r{L->desc[i].kv_group, L->desc[i].kind == LMC_LAYER_KDA};
            if (std::find(reads.begin(), reads.end(), r) == reads.end())
                reads.push_back(r);
        }
        for (int64_t q = 0; q < nj; q++) {
            const lmc_job &job = b->jobs[og][q];
            if (job.request < 0 || job.request >= b->num_requests || job.chunk < 0)
                continue;
            for (const auto &r : reads) {
                const lmc_block_table &t = b->tables[r.first];
                const int64_t first = (int64_t)job.chunk * pos_mul;
                const int64_t lo = r.second && !kda_every ? first + nb - 1 : first;
                for (int64_t p = lo; p < first + nb && p < t.num_cols; p++) {
                    const int32_t id = t.table[(int64_t)job.request * t.row_stride + p];
                    if (valid_block(id, L->num_blocks))
                        out.push_back(id);
                }
            }
        }
    }
    return LMC_OK;
}

}  // namespace

namespace lmc {

int check_copy_pairs(const lmc_layout *L, const lmc_copy_batch *b) {
    const int nkv = (int)L->kv_group_kind.size();
    if (b->host_pairs == nullptr)
        return LMC_ERR_INVALID_ARG;
    // (block, pair index) of every pair that moves data
    std::vector<std::pair<int32_t, int64_t>> dst;
    std::vector<std::pair<int32_t, int64_t>> src;
    int64_t index = 0;
    for (int g = 0; g < nkv; g++) {
        const int64_t n = b->num_pairs[g];
        if (n > 0 && b->host_pairs[g] == nullptr)
            return LMC_ERR_INVALID_ARG;
        for (int64_t q = 0; q < n; q++, index++) {
            const lmc_block_pair &p = b->host_pairs[g][q];
            if (!valid_block(p.src_block, L->num_blocks) || !valid_block(p.dst_block, L->num_blocks))
                continue;  // skipped by the kernel, with a status bit
            dst.emplace_back(p.dst_block, index);
            src.emplace_back(p.src_block, index);
        }
    }
    std::sort(dst.begin(), dst.end());
    for (size_t i = 1; i < dst.size(); i++)
        if (dst[i].first == dst[i - 1].first)
            return LMC_ERR_OVERLAP;  // one block written twice
    for (const auto &s : src) {
        const auto it = std::lower_bound(dst.begin(), dst.end(), std::make_pair(s.first, (int64_t)INT64_MIN));
        if (it != dst.end() && it->first == s.first && it->second != s.second)
            return LMC_ERR_OVERLAP;  // a block written by one pair and read by another
    }
    return LMC_OK;
}

}  // namespace lmc

namespace {

int disjoint(const lmc_layout *L, int64_t nb, int64_t pos_mul, bool kda_every, const lmc_batch *a,
             const lmc_batch *b, int32_t *out_block) {
    std::vector<int32_t> ta, tb;
    int rc = touched_blocks(L, nb, pos_mul, kda_every, a, ta);
    if (rc == LMC_OK)
        rc = touched_blocks(L, nb, pos_mul, kda_every, b, tb);
    if (rc != LMC_OK)
        return rc;
    std::sort(ta.begin(), ta.end());
    std::sort(tb.begin(), tb.end());
    std::vector<int32_t> common;
    std::set_intersection(ta.begin(), ta.end(), tb.begin(), tb.end(), std::back_inserter(common));
    if (out_block != nullptr)
        *out_block = common.empty() ? -1 : common.front();
    return common.empty() ? LMC_OK : LMC_ERR_OVERLAP;
}

}  // namespace

extern "C" int lmc_check_disjoint(const lmc_layout *L, int64_t chunk_size, const lmc_batch *a, const lmc_batch *b,
                                  int32_t *out_block) {
    if (L == nullptr || a == nullptr || b == nullptr)
        return LMC_ERR_INVALID_ARG;
    if (chunk_size <= 0 || chunk_size % L->block_size != 0)
        return LMC_ERR_NOT_MULTIPLE;
    const int64_t m = chunk_size / L->block_size;
    if (m > INT32_MAX)
        return LMC_ERR_OVERFLOW;
    return disjoint(L, m, m, false, a, b, out_block);
}

extern "C" int lmc_check_disjoint_blocks(const lmc_layout *L, int64_t blocks_per_object, int32_t kda_mode,
                                         const lmc_batch *a, const lmc_batch *b, int32_t *out_block) {
    if (L == nullptr || a == nullptr || b == nullptr || blocks_per_object <= 0 || blocks_per_object > INT32_MAX ||
        (kda_mode != LMC_KDA_LAST_BLOCK && kda_mode != LMC_KDA_EVERY_BLOCK))
        return LMC_ERR_INVALID_ARG;
    return disjoint(L, blocks_per_object, 1, kda_mode == LMC_KDA_EVERY_BLOCK, a, b, out_block);
}

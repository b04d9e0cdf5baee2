// lmc_internal.h -- the layout object shared by the host builder and the
// store/load launchers inside liblmc (not part of the public ABI).
#pragma once

#include <cstdint>
#include <vector>

#include "lmc.h"

struct lmc_layout {
    int64_t block_size = 0;
    int32_t mode = LMC_LAYOUT_PADDED;
    int32_t num_slabs = 0;
    int64_t page_size = 0;
    int64_t block_stride = 0;
    int64_t num_blocks = 0;
    int64_t pool_bytes = 0;
    std::vector<lmc_layer_spec> specs;      // model order
    std::vector<lmc_layer_desc> desc;       // model order
    std::vector<int32_t> kv_group_kind;
    std::vector<int32_t> kv_group_size;
    std::vector<int32_t> object_group_kind;
    // layers of each object group, in model order
    std::vector<std::vector<int32_t>> object_group_layers;
};

namespace lmc {

// Checked 64-bit arithmetic (false on overflow).
inline bool mul_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_mul_overflow(a, b, out); }
inline bool add_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_add_overflow(a, b, out); }

// The rule lmc_copy_blocks checks on the host copy of its pairs before any
// launch: among the pairs whose two block ids lie in the pool, no block is
// the destination of two pairs, nor the destination of one pair and the
// source of another (KV groups share block ids). LMC_OK or LMC_ERR_OVERLAP
// (LMC_ERR_INVALID_ARG when the host pairs are missing). The batch's group
// count and pair counts are checked by the caller.
int check_copy_pairs(const lmc_layout *L, const lmc_copy_batch *b);

}  // namespace lmc

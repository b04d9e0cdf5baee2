/* A plain C11 client of liblmc's host-side calls (no GPU needed): it checks
 * that include/lmc.h compiles as C and that the ABI works from C. It prints
 * "key value" lines that tests/test_c_abi.py compares with the Python
 * binding and with the values the pages give. */
#include <stdio.h>
#include <string.h>

#include "lmc.h"

static int fail(const char *what, int rc) {
    printf("error %s %d %s\n", what, rc, lmc_strerror(rc));
    return 1;
}

int main(void) {
    int64_t v = 0;
    int rc;

    /* unified block size: Kimi-Linear's 1152-byte MLA entry, TP 2 and TP 1 state pages */
    if ((rc = lmc_unified_block_size(1152, 73728 / 2 + 2097152 / 2, 16, &v)) != LMC_OK)
        return fail("unified_tp2", rc);
    printf("unified_tp2 %lld\n", (long long)v);
    if ((rc = lmc_unified_block_size(1152, 73728 + 2097152, 16, &v)) != LMC_OK)
        return fail("unified_tp1", rc);
    printf("unified_tp1 %lld\n", (long long)v);

    /* chunk negotiation and the strict rule */
    if ((rc = lmc_negotiate_chunk(100, 64, 0, &v)) != LMC_OK)
        return fail("negotiate", rc);
    printf("negotiate_100_64 %lld\n", (long long)v);
    printf("strict_100_64 %d\n", lmc_negotiate_chunk(100, 64, 1, &v));
    printf("negotiate_bad_n %d\n", lmc_negotiate_chunk(100, 0, 0, &v));

    /* scheduler budget */
    printf("budget_944_1887 %d\n", lmc_check_step_budget(944, 1887, 0));
    printf("budget_944_1888_joint %d\n", lmc_check_step_budget(944, 1888, 0));
    printf("budget_944_1888_separate %d\n", lmc_check_step_budget(944, 1888, 1));

    /* Kimi-Linear, 24 layers (KDA, KDA, KDA, MLA) x 6, N = 944, padded */
    lmc_layer_spec specs[24];
    memset(specs, 0, sizeof specs);
    for (int i = 0; i < 24; i++) {
        if (i % 4 == 3) {
            specs[i].kind = LMC_LAYER_MLA;
            specs[i].token_bytes = 1152;
        } else {
            specs[i].kind = LMC_LAYER_KDA;
            specs[i].conv_bytes = 73728;
            specs[i].rec_bytes = 2097152;
        }
    }
    lmc_layout_params p;
    memset(&p, 0, sizeof p);
    p.num_layers = 24;
    p.mode = LMC_LAYOUT_PADDED;
    p.grouping = LMC_GROUP_SPLIT;
    p.separate_object_groups = 1;
    p.block_size = 944;
    p.mem_bytes = (int64_t)1056 * 6 * 2170880;
    p.layers = specs;
    lmc_layout *L = NULL;
    if ((rc = lmc_layout_build(&p, &L)) != LMC_OK)
        return fail("layout_build", rc);
    lmc_layout_info info;
    if ((rc = lmc_layout_query(L, &info)) != LMC_OK)
        return fail("layout_query", rc);
    printf("num_kv_groups %d\n", info.num_kv_groups);
    printf("num_object_groups %d\n", info.num_object_groups);
    printf("num_slabs %d\n", info.num_slabs);
    printf("page_size %lld\n", (long long)info.page_size);
    printf("num_blocks %lld\n", (long long)info.num_blocks);
    printf("pool_bytes %lld\n", (long long)info.pool_bytes);
    for (int i = 0; i < info.num_layers; i++) {
        const lmc_layer_desc *d = &info.layers[i];
        printf("layer %d %d %d %d %d %lld %lld %lld %lld\n", i, d->kind, d->kv_group, d->slot, d->object_group,
               (long long)d->real_bytes, (long long)d->page_bytes, (long long)d->base, (long long)d->stride);
    }
    for (int g = 0; g < info.num_object_groups; g++) {
        if ((rc = lmc_object_bytes(L, 944, g, &v)) != LMC_OK)
            return fail("object_bytes", rc);
        printf("object_bytes %d %lld\n", g, (long long)v);
    }
    uint32_t bits = 0;
    if ((rc = lmc_layout_check_backends(L, 1, 0, &bits)) != LMC_OK)
        return fail("check_backends", rc);
    printf("backends_stride_attention %u\n", bits);

    /* host validation: a store without a batch is refused before any launch */
    printf("store_without_batch %d\n", lmc_store(L, 944, NULL, NULL, NULL, 0, NULL, NULL));
    printf("store_bad_chunk %d\n", lmc_store(L, 900, NULL, NULL, NULL, 0, NULL, NULL));
    printf("strerror_budget %s\n", lmc_strerror(LMC_ERR_BUDGET));
    lmc_layout_free(L);
    printf("done\n");
    return 0;
}

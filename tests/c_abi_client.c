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

    /* copy-on-write pairs that would race are refused on the host copy
     * before any launch (the pool pointer is NULL, so a batch that passed
     * the rule would be refused just before launching: nothing runs) */
    lmc_block_pair racing[2] = {{1, 9}, {9, 12}}; /* 9 written by one pair, read by the other */
    lmc_block_pair fine[2] = {{1, 9}, {2, 12}};
    const lmc_block_pair *dev_pairs[4] = {NULL, NULL, NULL, NULL};
    const lmc_block_pair *host_pairs[4] = {NULL, NULL, NULL, NULL};
    int64_t counts[4] = {0, 2, 0, 0};
    lmc_copy_batch cb;
    memset(&cb, 0, sizeof cb);
    cb.num_kv_groups = info.num_kv_groups;
    cb.pairs = dev_pairs;
    cb.num_pairs = counts;
    cb.host_pairs = host_pairs;
    dev_pairs[1] = racing; /* never dereferenced on the host */
    host_pairs[1] = racing;
    uint32_t status_word = 0;
    printf("copy_racing %d\n", lmc_copy_blocks(L, NULL, &cb, &status_word, NULL));
    dev_pairs[1] = fine;
    host_pairs[1] = fine;
    printf("copy_fine_null_pool %d\n", lmc_copy_blocks(L, NULL, &cb, &status_word, NULL));
    cb.host_pairs = NULL;
    printf("copy_without_host_pairs %d\n", lmc_copy_blocks(L, NULL, &cb, &status_word, NULL));

    /* mixed-step guard on host arrays (chunk = N, one request): the load
     * side moves chunk 0, whose position 0 holds blocks 0, 10, 20, 30 in
     * the four KV groups' tables; the store side chunk 1 of other tables
     * (blocks 6, 16, 26, 36) */
    int32_t tables_a[4][2], tables_b[4][2];
    lmc_block_table ta[4], tb[4];
    for (int k = 0; k < 4; k++) {
        tables_a[k][0] = 10 * k;
        tables_a[k][1] = 10 * k + 1;
        tables_b[k][0] = 10 * k + 5;
        tables_b[k][1] = 10 * k + 6;
        ta[k].table = tables_a[k];
        tb[k].table = tables_b[k];
        ta[k].row_stride = tb[k].row_stride = 2;
        ta[k].num_cols = tb[k].num_cols = 2;
    }
    lmc_job ja = {0, 0, 0}, jb = {0, 1, 0};
    const lmc_job *jobs_a[2] = {&ja, &ja}, *jobs_b[2] = {&jb, &jb};
    int64_t njobs[2] = {1, 1};
    lmc_batch ba = {1, 4, ta, 2, 0, jobs_a, njobs}, bb = {1, 4, tb, 2, 0, jobs_b, njobs};
    int32_t common = 0;
    rc = lmc_check_disjoint(L, 944, &ba, &bb, &common);
    printf("disjoint %d %d\n", rc, common);
    tables_b[2][1] = 20; /* the store side now reads block 20, which the load side writes */
    rc = lmc_check_disjoint(L, 944, &ba, &bb, &common);
    printf("shared %d %d\n", rc, common);
    lmc_layout_free(L);
    printf("done\n");
    return 0;
}

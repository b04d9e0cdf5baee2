/* A plain C11 client of liblmc's device calls: it reads a workload written by
 * tests/test_c_abi.py (layer specs, block tables, jobs, pool bytes), moves it
 * with lmc_store / lmc_load through the C ABI on the default stream using
 * device memory from the CUDA runtime's C API, and writes the arena and the
 * reloaded pool back for the test to compare with the oracle.
 *
 * usage: c_abi_gpu_client DIR
 *   DIR/case.txt   "N packed mem chunk requests cols layers kv_groups object_groups"
 *                  then one line per layer "kind token_bytes conv_bytes rec_bytes window",
 *                  then one line per object group "num_jobs", then "arena_bytes"
 *   DIR/pool.bin, DIR/src_K.bin, DIR/dst_K.bin (int32 [requests][cols]), DIR/jobs_G.bin
 * writes DIR/arena.out, DIR/fresh.out, DIR/status.out */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "lmc.h"

static void *read_file(const char *dir, const char *name, size_t *size) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f)
        return NULL;
    fseek(f, 0, SEEK_END);
    long n = ftell(f);
    fseek(f, 0, SEEK_SET);
    void *buf = malloc(n > 0 ? (size_t)n : 1);
    if (buf && n > 0 && fread(buf, 1, (size_t)n, f) != (size_t)n) {
        free(buf);
        buf = NULL;
    }
    fclose(f);
    *size = (size_t)n;
    return buf;
}

static int write_file(const char *dir, const char *name, const void *data, size_t n) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f)
        return 1;
    size_t w = fwrite(data, 1, n, f);
    fclose(f);
    return w != n;
}

static void *to_device(const void *host, size_t n) {
    void *d = NULL;
    if (cudaMalloc(&d, n ? n : 16) != cudaSuccess)
        return NULL;
    if (n && cudaMemcpy(d, host, n, cudaMemcpyHostToDevice) != cudaSuccess)
        return NULL;
    return d;
}

#define CHECK(cond, what)                         \
    do {                                          \
        if (!(cond)) {                            \
            fprintf(stderr, "failed: %s\n", what); \
            return 1;                             \
        }                                         \
    } while (0)

int main(int argc, char **argv) {
    CHECK(argc == 2, "usage: c_abi_gpu_client DIR");
    const char *dir = argv[1];
    char path[4096];
    snprintf(path, sizeof path, "%s/case.txt", dir);
    FILE *f = fopen(path, "r");
    CHECK(f != NULL, "case.txt");
    long long N, packed, mem, chunk, requests, cols, layers, kv_groups, object_groups, arena_bytes;
    CHECK(fscanf(f, "%lld %lld %lld %lld %lld %lld %lld %lld %lld", &N, &packed, &mem, &chunk, &requests, &cols,
                 &layers, &kv_groups, &object_groups) == 9,
          "case header");
    CHECK(layers > 0 && layers <= LMC_MAX_LAYERS && kv_groups > 0 && kv_groups <= 64 && object_groups > 0 &&
              object_groups <= 64,
          "case sizes");
    lmc_layer_spec specs[LMC_MAX_LAYERS];
    memset(specs, 0, sizeof specs);
    for (long long i = 0; i < layers; i++) {
        long long kind, tb, conv, rec, window;
        CHECK(fscanf(f, "%lld %lld %lld %lld %lld", &kind, &tb, &conv, &rec, &window) == 5, "layer line");
        specs[i].kind = (int32_t)kind;
        specs[i].token_bytes = tb;
        specs[i].conv_bytes = conv;
        specs[i].rec_bytes = rec;
        specs[i].window = (int32_t)window;
    }
    int64_t num_jobs[64];
    for (long long g = 0; g < object_groups; g++) {
        long long n;
        CHECK(fscanf(f, "%lld", &n) == 1, "job count");
        num_jobs[g] = n;
    }
    CHECK(fscanf(f, "%lld", &arena_bytes) == 1, "arena bytes");
    fclose(f);

    lmc_layout_params p;
    memset(&p, 0, sizeof p);
    p.num_layers = (int32_t)layers;
    p.mode = packed ? LMC_LAYOUT_PACKED : LMC_LAYOUT_PADDED;
    p.grouping = LMC_GROUP_SPLIT;
    p.separate_object_groups = 1;
    p.block_size = N;
    p.mem_bytes = mem;
    p.layers = specs;
    lmc_layout *L = NULL;
    CHECK(lmc_layout_build(&p, &L) == LMC_OK, "lmc_layout_build");
    lmc_layout_info info;
    CHECK(lmc_layout_query(L, &info) == LMC_OK, "lmc_layout_query");
    CHECK(info.num_kv_groups == kv_groups && info.num_object_groups == object_groups, "group counts");

    size_t pool_n = 0, n = 0;
    void *pool_h = read_file(dir, "pool.bin", &pool_n);
    CHECK(pool_h != NULL && (int64_t)pool_n == info.pool_bytes, "pool.bin");
    void *pool = to_device(pool_h, pool_n);
    void *fresh_h = malloc(pool_n);
    CHECK(fresh_h != NULL, "malloc");
    memset(fresh_h, 0xA5, pool_n);
    void *fresh = to_device(fresh_h, pool_n);
    void *arena = NULL;
    CHECK(cudaMalloc(&arena, (size_t)arena_bytes) == cudaSuccess, "cudaMalloc arena");
    CHECK(cudaMemset(arena, 0x3C, (size_t)arena_bytes) == cudaSuccess, "cudaMemset arena");
    uint32_t *status = NULL;
    CHECK(cudaMalloc((void **)&status, 4) == cudaSuccess && cudaMemset(status, 0, 4) == cudaSuccess, "status");

    lmc_block_table src_t[64], dst_t[64];
    for (long long k = 0; k < kv_groups; k++) {
        char name[64];
        snprintf(name, sizeof name, "src_%lld.bin", k);
        void *h = read_file(dir, name, &n);
        CHECK(h != NULL && n == (size_t)(requests * cols * 4), "src table");
        src_t[k].table = (const int32_t *)to_device(h, n);
        src_t[k].row_stride = cols;
        src_t[k].num_cols = cols;
        free(h);
        snprintf(name, sizeof name, "dst_%lld.bin", k);
        h = read_file(dir, name, &n);
        CHECK(h != NULL && n == (size_t)(requests * cols * 4), "dst table");
        dst_t[k].table = (const int32_t *)to_device(h, n);
        dst_t[k].row_stride = cols;
        dst_t[k].num_cols = cols;
        free(h);
    }
    const lmc_job *jobs[64];
    for (long long g = 0; g < object_groups; g++) {
        char name[64];
        snprintf(name, sizeof name, "jobs_%lld.bin", g);
        void *h = read_file(dir, name, &n);
        CHECK(h != NULL && n == (size_t)num_jobs[g] * sizeof(lmc_job), "jobs");
        jobs[g] = (const lmc_job *)to_device(h, n);
        free(h);
    }
    lmc_batch b;
    memset(&b, 0, sizeof b);
    b.num_requests = (int32_t)requests;
    b.num_kv_groups = (int32_t)kv_groups;
    b.num_object_groups = (int32_t)object_groups;
    b.jobs = jobs;
    b.num_jobs = num_jobs;

    b.tables = src_t;
    CHECK(lmc_store(L, chunk, pool, &b, arena, arena_bytes, status, NULL) == LMC_OK, "lmc_store");
    b.tables = dst_t;
    CHECK(lmc_load(L, chunk, fresh, &b, arena, arena_bytes, status, NULL) == LMC_OK, "lmc_load");
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "synchronize");

    void *arena_h = malloc((size_t)arena_bytes);
    uint32_t st = 0;
    CHECK(arena_h != NULL, "malloc");
    CHECK(cudaMemcpy(arena_h, arena, (size_t)arena_bytes, cudaMemcpyDeviceToHost) == cudaSuccess, "arena back");
    CHECK(cudaMemcpy(fresh_h, fresh, pool_n, cudaMemcpyDeviceToHost) == cudaSuccess, "pool back");
    CHECK(cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost) == cudaSuccess, "status back");
    CHECK(write_file(dir, "arena.out", arena_h, (size_t)arena_bytes) == 0, "arena.out");
    CHECK(write_file(dir, "fresh.out", fresh_h, pool_n) == 0, "fresh.out");
    char sbuf[32];
    snprintf(sbuf, sizeof sbuf, "%u\n", st);
    CHECK(write_file(dir, "status.out", sbuf, strlen(sbuf)) == 0, "status.out");
    lmc_layout_free(L);
    printf("done\n");
    return 0;
}

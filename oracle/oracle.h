/*
 * oracle.h -- declarations of the CPU oracle (test infrastructure only).
 * The product library has its own header and never includes this one.
 */
#ifndef STATE_CACHE_PAGING_ORACLE_H
#define STATE_CACHE_PAGING_ORACLE_H

#include <stdint.h>

#define OR_MAX_LAYERS 256

/* Return codes (same numeric meaning as the library's, written separately). */
#define OR_OK 0
#define OR_ERR_INVALID_ARG (-1)
#define OR_ERR_ALIGN (-2)
#define OR_ERR_NOT_MULTIPLE (-3)
#define OR_ERR_NO_MEMORY (-4)
#define OR_ERR_OVERFLOW (-6)
#define OR_ERR_BUDGET (-7)
#define OR_ERR_OVERLAP (-8)

/* Status bits raised by a store or load; the offending page is skipped. */
#define OR_ST_BLOCK_OOR 0x1u   /* block id outside [0, num_blocks), not -1 */
#define OR_ST_NO_BLOCK 0x2u    /* -1 where a paged attention block is needed */
#define OR_ST_NO_SNAPSHOT 0x4u /* -1 where a KDA snapshot is needed */
#define OR_ST_BAD_JOB 0x8u     /* bad request/chunk/offset, or past the table */

/* Backend-eligibility bits. */
#define OR_BK_PADDED_ATTENTION 0x1u /* an attention page is padded, backend cannot stride */
#define OR_BK_PACKED_ATTENTION 0x2u /* packed, an attention backend cannot stride */
#define OR_BK_PACKED_STATE 0x4u     /* packed, a state (KDA) kernel needs contiguous pages */

/* Layer kinds. */
#define OR_MLA 0
#define OR_KDA 1
#define OR_SWA 2

typedef struct {
    int32_t kind;
    int32_t window;      /* sliding-window tokens (SWA only) */
    int64_t token_bytes; /* bytes per token of a paged attention layer */
    int64_t conv_bytes;  /* KDA conv_state bytes */
    int64_t rec_bytes;   /* KDA recurrent_state bytes */
} or_layer;

typedef struct {
    /* inputs */
    int32_t num_layers;
    int32_t packed;                 /* 0: padded (path A), 1: packed (path B) */
    int32_t split_groups;           /* 1: near-equal runs per spec, 0: one group per spec */
    int32_t separate_object_groups; /* 1: one object group per window class */
    int64_t N;                      /* block size in tokens */
    int64_t mem_bytes;              /* memory offered to the pool */
    or_layer layers[OR_MAX_LAYERS];
    /* results */
    int32_t num_kv_groups;
    int32_t num_object_groups;
    int32_t num_slabs;
    int32_t pad_;
    int64_t page_size;    /* padded: the unified page; packed: 0 */
    int64_t block_stride; /* bytes from block b to block b+1 of one layer */
    int64_t num_blocks;
    int64_t pool_bytes;
    int32_t kv_group[OR_MAX_LAYERS];
    int32_t slot[OR_MAX_LAYERS]; /* position of the layer inside its KV group */
    int32_t object_group[OR_MAX_LAYERS];
    int32_t kv_group_kind[OR_MAX_LAYERS];
    int32_t kv_group_size[OR_MAX_LAYERS];
    int64_t real_bytes[OR_MAX_LAYERS];
    int64_t page_bytes[OR_MAX_LAYERS];
    int64_t base[OR_MAX_LAYERS];   /* pool byte offset of block 0's page */
    int64_t stride[OR_MAX_LAYERS]; /* bytes between consecutive blocks' pages */
} or_layout;

typedef struct {
    int32_t request;
    int32_t chunk;
    int64_t offset; /* byte offset of the object in the arena */
} or_job;

typedef struct {
    int32_t num_requests;
    int32_t num_kv_groups;
    const int32_t *const *table; /* [kv group] -> [num_requests][row_stride] */
    const int64_t *row_stride;   /* [kv group] */
    const int64_t *num_cols;     /* [kv group] valid block positions per row */
} or_tables;

typedef struct {
    int32_t num_object_groups;
    int32_t pad_;
    const or_job *const *jobs; /* [object group] -> job array */
    const int64_t *num_jobs;   /* [object group] */
} or_jobs;

typedef struct {
    int64_t pool_offset;
    int64_t object_offset;
    int64_t bytes;
    int32_t layer;
    int32_t block;
} or_page;

typedef struct {
    or_page *pages;
    int64_t capacity;
    int64_t count;
} or_page_list;

int or_negotiate_chunk(int64_t requested, int64_t N, int strict, int64_t *out);
int or_check_step_budget(int64_t N, int64_t max_batched, int separate_object_groups);
int or_layout_build(or_layout *L);
uint32_t or_check_backends(const or_layout *L, int attn_indexes_by_stride, int state_pages_strided_ok);
int64_t or_object_bytes(const or_layout *L, int64_t C, int og);
int or_store(const or_layout *L, int64_t C, const uint8_t *pool,
             const or_tables *T, const or_jobs *J,
             uint8_t *arena, int64_t arena_bytes, uint32_t *status);
int or_load(const or_layout *L, int64_t C, uint8_t *pool,
            const or_tables *T, const or_jobs *J,
            const uint8_t *arena, int64_t arena_bytes, uint32_t *status);

int or_list_pages(const or_layout *L, int64_t C, const or_tables *T, const or_jobs *J,
                  int64_t arena_bytes, uint32_t *status, or_page_list *list);
int or_list_pages_any(const or_layout *L, int64_t C, int64_t nb, int kda_every,
                      const or_tables *T, const or_jobs *J,
                      int64_t arena_bytes, uint32_t *status, or_page_list *list);
int64_t or_object_bytes_blocks(const or_layout *L, int64_t nb, int kda_every, int og);
int or_store_blocks(const or_layout *L, int64_t nb, int kda_every, const uint8_t *pool,
                    const or_tables *T, const or_jobs *J,
                    uint8_t *arena, int64_t arena_bytes, uint32_t *status);
int or_load_blocks(const or_layout *L, int64_t nb, int kda_every, uint8_t *pool,
                   const or_tables *T, const or_jobs *J,
                   const uint8_t *arena, int64_t arena_bytes, uint32_t *status);

typedef struct {
    int32_t src_block;
    int32_t dst_block;
} or_pair;

typedef struct {
    int32_t num_kv_groups;
    int32_t pad_;
    const or_pair *const *pairs; /* [kv group] -> pair array */
    const int64_t *num_pairs;    /* [kv group] */
} or_copy_batch;

int or_copy_blocks(const or_layout *L, uint8_t *pool, const or_copy_batch *B, uint32_t *status);
int or_check_disjoint(const or_layout *L, int64_t C, const or_tables *Ta, const or_jobs *Ja,
                      const or_tables *Tb, const or_jobs *Jb, int32_t *out_block);
int or_check_disjoint_blocks(const or_layout *L, int64_t nb, int kda_every, const or_tables *Ta,
                             const or_jobs *Ja, const or_tables *Tb, const or_jobs *Jb, int32_t *out_block);

int or_store_q8(const or_layout *L, int64_t C, int64_t d, const uint8_t *pool,
                const or_tables *T, const or_jobs *J,
                uint8_t *arena, int64_t arena_bytes, uint32_t *status);
int or_load_q8(const or_layout *L, int64_t C, int64_t d, uint8_t *pool,
               const or_tables *T, const or_jobs *J,
               const uint8_t *arena, int64_t arena_bytes, uint32_t *status);
int64_t or_object_bytes_q8(const or_layout *L, int64_t C, int64_t d, int og);
int or_store_blocks_q8(const or_layout *L, int64_t nb, int kda_every, int64_t d, const uint8_t *pool,
                       const or_tables *T, const or_jobs *J,
                       uint8_t *arena, int64_t arena_bytes, uint32_t *status);
int or_load_blocks_q8(const or_layout *L, int64_t nb, int kda_every, int64_t d, uint8_t *pool,
                      const or_tables *T, const or_jobs *J,
                      const uint8_t *arena, int64_t arena_bytes, uint32_t *status);
int64_t or_object_bytes_blocks_q8(const or_layout *L, int64_t nb, int kda_every, int64_t d, int og);
int or_unified_block_size(int64_t attn_token_bytes, int64_t state_page_bytes,
                          int64_t align, int64_t *out);

#endif

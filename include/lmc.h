/*
 * lmc.h -- C ABI of liblmc: paging a hybrid KDA (linear attention) + MLA
 * model's cache between a vLLM-style paged GPU pool and LMCache-style
 * per-chunk objects, on one GB300 (sm_103a).
 *
 * Sources (page title, section):
 *   [KL] "Kimi-Linear" (LMCache recipe): unified block size N, chunk size a
 *        multiple of N, scheduler budget in [N, 2N), KDA state snapshots at
 *        block boundaries, cached pages are byte-opaque.
 *   [K3] "Kimi K3" (LMCache recipe): --chunk-size is a minimum that is
 *        negotiated to the smallest multiple of N at or above it.
 *   [VB] "How vLLM manages the KV cache of hybrid models: Kimi Linear / Kimi
 *        K3" (blog): §2.1 KDA state shapes, §2.2 KV cache groups, §3.1 the
 *        padded shared-tensor layout (path A), §3.2 the packed layout
 *        (path B), §4 the int8 buffer and its per-layer views.
 *   [MC] "When Prefix Cache Meets KDA" (Mooncake post): checkpoints must sit
 *        on a prefix boundary shared by MLA KV and KDA state; "Flat KV": 69
 *        KDA layers in three groups of 23 plus the full-attention group on
 *        24 physical slabs.
 *   [HM] "Hybrid Attention Models" (LMCache docs): "Object-group
 *        separation" (one object per chunk and attention window class),
 *        Step 1 / Step 2 (N, chunk size, budget).
 *
 * Conventions for every call:
 *   - Return value: LMC_OK (0) or a negative LMC_ERR_* code. Argument errors
 *     are found on the host before anything is enqueued; on error nothing is
 *     enqueued and no output is touched.
 *   - Device-side problems found while copying (a bad block id, a missing
 *     snapshot, a bad job) do not stop the launch: the page or object
 *     concerned is skipped and an LMC_ST_* bit is OR-ed into the caller's
 *     device status word, which the caller reads after synchronising.
 *   - Ownership: the caller owns all device memory (pool, block tables, jobs,
 *     arena, status word). The library allocates no device memory, never
 *     synchronises, and reads host-side structs only during the call.
 *   - Streams: store/load are asynchronous on the given cudaStream_t (passed
 *     as void*; NULL is the legacy default stream).
 *   - Thread safety: a built layout is immutable and may be shared by
 *     threads and streams. Calls that write overlapping memory on different
 *     streams race.
 */
#ifndef LMC_H
#define LMC_H

#include <stdint.h>

/* Only the lmc_* entry points are exported from liblmc.so. */
#if defined(__GNUC__)
#define LMC_API __attribute__((visibility("default")))
#else
#define LMC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------- */
#define LMC_OK 0
#define LMC_ERR_INVALID_ARG (-1)  /* NULL pointer, bad size, inconsistent batch */
#define LMC_ERR_ALIGN (-2)        /* status word not 4-byte aligned */
#define LMC_ERR_NOT_MULTIPLE (-3) /* chunk not a positive multiple of N */
#define LMC_ERR_NO_MEMORY (-4)    /* mem_bytes below one block of the layout */
#define LMC_ERR_CUDA (-5)         /* a CUDA runtime call failed */
#define LMC_ERR_OVERFLOW (-6)     /* a size does not fit 64-bit arithmetic */
#define LMC_ERR_BUDGET (-7)       /* scheduler budget outside the allowed range */
#define LMC_ERR_OVERLAP (-8)      /* copies that would race: a block written twice, or
                                     written by one copy and read by another */

/* ---- device status bits (OR-ed into *status) ----------------------------- */
#define LMC_ST_BLOCK_OOR 0x1u   /* block id < -1 or >= num_blocks */
#define LMC_ST_NO_BLOCK 0x2u    /* -1 where a paged attention block is needed */
#define LMC_ST_NO_SNAPSHOT 0x4u /* -1 where a KDA state snapshot is needed */
#define LMC_ST_BAD_JOB 0x8u     /* request out of range, chunk < 0, block position
                                   past the table's columns, or an object that is
                                   not 16-byte aligned or does not fit the arena */
#define LMC_ST_TIMEOUT 0x10u    /* a bounded wait inside the kernel gave up; the
                                   launch's output is incomplete */

/* ---- layer specs --------------------------------------------------------- */
#define LMC_LAYER_MLA 0 /* full attention, one latent entry per token */
#define LMC_LAYER_KDA 1 /* linear attention: conv_state + recurrent_state */
#define LMC_LAYER_SWA 2 /* sliding-window paged attention */

#define LMC_LAYOUT_PADDED 0 /* [VB] §3.1 path A */
#define LMC_LAYOUT_PACKED 1 /* [VB] §3.2 path B */

#define LMC_GROUP_SPLIT 0   /* equal-spec layers split into near-equal runs
                               (run count = ceil(count / smallest count)) */
#define LMC_GROUP_BY_SPEC 1 /* one KV cache group per distinct spec ([VB] §2.2) */

#define LMC_MAX_LAYERS 256

typedef struct {
    int32_t kind;        /* LMC_LAYER_* */
    int32_t window;      /* SWA window in tokens (> 0); 0 for other kinds */
    int64_t token_bytes; /* MLA/SWA: bytes of one token's cache entry
                            (e.g. (512 + 64) bf16 latent = 1152) */
    int64_t conv_bytes;  /* KDA: bytes of conv_state (conv_dim, k - 1) */
    int64_t rec_bytes;   /* KDA: bytes of recurrent_state (heads, d, d) */
} lmc_layer_spec;

typedef struct {
    int32_t num_layers;             /* 1 .. LMC_MAX_LAYERS, model order */
    int32_t mode;                   /* LMC_LAYOUT_PADDED or LMC_LAYOUT_PACKED */
    int32_t grouping;               /* LMC_GROUP_SPLIT or LMC_GROUP_BY_SPEC */
    int32_t separate_object_groups; /* 1: one object group per window class
                                       (full attention, KDA, each SWA window);
                                       0: a single object group ([HM]) */
    int64_t block_size;             /* N, tokens per block (> 0) */
    int64_t mem_bytes;              /* memory offered to the pool */
    const lmc_layer_spec *layers;   /* host array [num_layers]; layers whose
                                       specs are equal in every field share a
                                       spec bucket when forming KV groups */
} lmc_layout_params;

typedef struct lmc_layout lmc_layout; /* opaque, immutable once built */

/* Per-layer address descriptor: block b of layer i starts at pool byte
 * base + b * stride and holds real_bytes of data (page_bytes allocated). */
typedef struct {
    int32_t kind;
    int32_t kv_group;     /* KV cache group: owns one block table */
    int32_t slot;         /* index of the layer inside its KV group */
    int32_t object_group; /* object group the layer's bytes are stored in */
    int64_t real_bytes;   /* MLA/SWA: N * token_bytes; KDA: conv + rec */
    int64_t page_bytes;   /* padded: the unified page size; packed: real_bytes */
    int64_t base;
    int64_t stride;
} lmc_layer_desc;

typedef struct {
    int32_t num_layers;
    int32_t num_kv_groups;
    int32_t num_object_groups;
    int32_t num_slabs;      /* largest KV group (path A: number of shared tensors) */
    int64_t block_size;     /* N */
    int64_t page_size;      /* padded: max real page; packed: 0 */
    int64_t block_stride;   /* padded: page_size; packed: max group byte total */
    int64_t num_blocks;     /* padded: mem // (num_slabs * page_size);
                               packed: mem // block_stride */
    int64_t pool_bytes;     /* bytes of the pool the descriptors address */
    const lmc_layer_desc *layers;  /* [num_layers], owned by the layout */
    const int32_t *kv_group_kind;  /* [num_kv_groups] LMC_LAYER_* */
    const int32_t *kv_group_size;  /* [num_kv_groups] layers per group */
    const int32_t *object_group_kind; /* [num_object_groups] kind of the
                                         group's first layer */
} lmc_layout_info;

/* Builds the pool layout ([VB] §2.2 grouping, §3.1 padded / §3.2 packed, §4
 * byte-opaque views; [MC] "Flat KV" slab count). Padded: page_size = the
 * largest real page, slab t (page_size * num_blocks bytes) is shared by the
 * t-th layer of every KV group, base = t * page_size * num_blocks,
 * stride = page_size. Packed: inside each KV group the layers' real pages are
 * laid back to back (cumulative offsets in model order), block_stride = the
 * largest group total, base = offset, stride = block_stride.
 * *out receives a layout owned by the caller (free with lmc_layout_free).
 * Errors: INVALID_ARG (bad spec), NO_MEMORY (not one whole block), OVERFLOW. */
LMC_API int lmc_layout_build(const lmc_layout_params *params, lmc_layout **out);

/* Fills *out with the layout's geometry; the arrays point into the layout and
 * live until lmc_layout_free. */
LMC_API int lmc_layout_query(const lmc_layout *layout, lmc_layout_info *out);

/* Frees a layout (NULL is ignored). No call using it may still be running. */
LMC_API void lmc_layout_free(lmc_layout *layout);

/* Backend-eligibility bits of lmc_layout_check_backends. */
#define LMC_BK_PADDED_ATTENTION 0x1u /* padded path pads an attention page, but the
                                        attention backend cannot index by block stride */
#define LMC_BK_PACKED_ATTENTION 0x2u /* packed path, an attention backend cannot stride */
#define LMC_BK_PACKED_STATE 0x4u     /* packed path, a state (KDA) kernel needs
                                        contiguous pages */

/* Which kernels can read the layout ([VB] §3.3): padding an attention layer's
 * page needs an attention backend that indexes pages by the block stride
 * (vLLM raises otherwise); the packed path needs every backend to address
 * pages by the block stride, and KDA kernels that assume contiguous pages
 * (causal_conv1d, chunk_kda) cannot, so such models fall back to the padded
 * path. *out_bits gets the LMC_BK_* bits of every rule broken (0: readable).
 * The store/load calls themselves work on any layout. */
LMC_API int lmc_layout_check_backends(const lmc_layout *layout, int attn_indexes_by_stride, int state_pages_strided_ok,
                              uint32_t *out_bits);

/* Bytes of one object of `object_group` for chunk size `chunk` ([HM] object
 * groups): the group's layers in model order, a paged layer contributing its
 * chunk / N pages of real_bytes (the chunk's tokens in order), a KDA layer one
 * state snapshot of real_bytes. Error NOT_MULTIPLE if chunk is not a positive
 * multiple of N. */
LMC_API int lmc_object_bytes(const lmc_layout *layout, int64_t chunk, int32_t object_group,
                     int64_t *out);

/* Chunk-size negotiation ([K3] "Chunk-Size Negotiation"): *out = the smallest
 * multiple of block_size at or above `requested` (block_size itself when
 * requested <= 0). strict != 0 applies the older rule ([KL], [HM] Step 2):
 * `requested` must already be a positive multiple of block_size, else
 * NOT_MULTIPLE (INVALID_ARG when requested <= 0). Errors: INVALID_ARG when
 * block_size <= 0 or out is NULL, OVERFLOW. */
LMC_API int lmc_negotiate_chunk(int64_t requested, int64_t block_size, int strict, int64_t *out);

/* Scheduler budget rule ([KL] "Why these settings", [HM] Step 2): OK when
 * N <= max_batched < 2N, or max_batched >= 2N with separate object groups;
 * BUDGET otherwise; INVALID_ARG for non-positive arguments. */
LMC_API int lmc_check_step_budget(int64_t block_size, int64_t max_batched, int separate_object_groups);

/* Smallest multiple of `align` tokens whose attention page
 * (N * attn_token_bytes) is at least `state_page_bytes` ([HM] Step 1, [KL]
 * note on N). With Kimi-Linear's 1152-byte MLA entry and align 16 this gives
 * 944 for the TP-2 state page and 1888 for TP 1. */
LMC_API int lmc_unified_block_size(int64_t attn_token_bytes, int64_t state_page_bytes, int64_t align,
                           int64_t *out);

/* ---- store / load -------------------------------------------------------- */

/* One object to move: chunk `chunk` of request `request`, at byte `offset` of
 * the arena (a multiple of 16). 16 bytes, device memory. */
typedef struct {
    int32_t request;
    int32_t chunk;
    int64_t offset;
} lmc_job;

/* One KV group's block table: int32 device matrix [num_requests][row_stride];
 * entry (r, p) is the block holding block position p (tokens [p*N, (p+1)*N))
 * of request r, or -1. For a KDA group, position p holds the state snapshot
 * taken after (p+1)*N tokens ([KL], [VB] §7 align mode). */
typedef struct {
    const int32_t *table;
    int64_t row_stride; /* elements between rows (>= num_cols) */
    int64_t num_cols;   /* valid positions per row */
} lmc_block_table;

typedef struct {
    int32_t num_requests;
    int32_t num_kv_groups;          /* must equal the layout's */
    const lmc_block_table *tables;  /* host array [num_kv_groups] */
    int32_t num_object_groups;      /* must equal the layout's */
    int32_t reserved;               /* set to 0 */
    const lmc_job *const *jobs;     /* host array [num_object_groups] of device
                                       pointers (NULL allowed when the count is 0) */
    const int64_t *num_jobs;        /* host array [num_object_groups] */
} lmc_batch;

/* Store (gather): for every job of every object group, writes the object
 * into arena + offset: for each layer of the group in model order, a paged
 * layer's blocks at positions chunk*m .. chunk*m + m - 1 (m = chunk_size / N)
 * copied back to back (token-major), a KDA layer's snapshot at position
 * (chunk + 1) * m - 1, the state at the chunk's end ([KL] snapshots at block
 * boundaries; [MC] restores resume only from a boundary checkpoint).
 * Only real bytes are copied; padding is never read. A launch handles layouts
 * of up to 64 KV groups and 64 object groups (INVALID_ARG beyond).
 * pool: device, >= pool_bytes, read only. arena: device, arena_bytes bytes.
 * status: device uint32, 4-byte aligned; bits are OR-ed, never cleared.
 * Errors (host): INVALID_ARG, NOT_MULTIPLE, ALIGN, CUDA (launch failure). */
LMC_API int lmc_store(const lmc_layout *layout, int64_t chunk_size, const void *pool,
              const lmc_batch *batch, void *arena, int64_t arena_bytes, uint32_t *status,
              void *stream);

/* Load (scatter): the exact inverse of lmc_store under the batch's block
 * tables, typically freshly allocated blocks of another pool ([VB] §5.3 a
 * hit's state becomes the initial state; [MC] restore at a checkpoint).
 * Writes only the real bytes of the addressed pages; every other pool byte
 * is left as it was. Same arguments and errors as lmc_store. */
LMC_API int lmc_load(const lmc_layout *layout, int64_t chunk_size, void *pool,
             const lmc_batch *batch, const void *arena, int64_t arena_bytes, uint32_t *status,
             void *stream);

/* ---- block-granular objects ---------------------------------------------- */

/* How a block-granular object holds KDA state. */
#define LMC_KDA_LAST_BLOCK 0  /* one snapshot: the object's last block */
#define LMC_KDA_EVERY_BLOCK 1 /* one snapshot per block of the object, in order */

/* Bytes of one block-granular object of `object_group` covering
 * `blocks_per_object` blocks: paged layers hold all blocks' pages, KDA layers
 * one snapshot (LMC_KDA_LAST_BLOCK) or one per block (LMC_KDA_EVERY_BLOCK).
 * With blocks_per_object = chunk / N and LMC_KDA_LAST_BLOCK this equals
 * lmc_object_bytes. Error INVALID_ARG for blocks_per_object <= 0 or an
 * unknown kda_mode. */
LMC_API int lmc_object_bytes_blocks(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                            int32_t object_group, int64_t *out);

/* Block-granular store/load: like lmc_store/lmc_load, but each job's `chunk`
 * field is the object's FIRST BLOCK POSITION and every object covers
 * `blocks_per_object` consecutive positions. This stores the whole blocks
 * past a request's last whole chunk (a tail object), objects aligned to
 * scheduler steps rather than chunks ([KL] "Why these settings": a step of
 * >= 2N tokens snapshots only its last block), and, with
 * LMC_KDA_EVERY_BLOCK, the snapshots of every block boundary inside an
 * object ([KL] the [N, 2N) regime; [VB] §7). Same arguments, ownership,
 * status bits and errors as lmc_store/lmc_load otherwise. */
LMC_API int lmc_store_blocks(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                     const void *pool, const lmc_batch *batch, void *arena, int64_t arena_bytes,
                     uint32_t *status, void *stream);
LMC_API int lmc_load_blocks(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode, void *pool,
                    const lmc_batch *batch, const void *arena, int64_t arena_bytes, uint32_t *status,
                    void *stream);

/* ---- in-pool block copies ------------------------------------------------ */

/* One copy: every layer page of a KV group, from block src to block dst. */
typedef struct {
    int32_t src_block;
    int32_t dst_block;
} lmc_block_pair;

typedef struct {
    int32_t num_kv_groups;            /* must equal the layout's */
    int32_t reserved;                 /* set to 0 */
    const lmc_block_pair *const *pairs; /* host array [num_kv_groups] of device
                                           pointers (NULL allowed when the count is 0) */
    const int64_t *num_pairs;         /* host array [num_kv_groups] */
    const lmc_block_pair *const *host_pairs; /* host array [num_kv_groups] of HOST
                                           pointers to the same pairs as `pairs`
                                           (the copy the caller built them from;
                                           NULL allowed when the count is 0): the
                                           call checks the pairs on them */
} lmc_copy_batch;

/* In-pool copies ([MC] "Copy-on-Write": a hit's shared KDA checkpoint is
 * copied into a private execution slot before it is updated; "Snapshot": a
 * running state is copied into a spare buffer at a cacheable boundary).
 * For each pair of KV group g, the real bytes of every layer of g are copied
 * from block src_block to block dst_block of `pool` (padding untouched).
 * A request's whole KDA state is one pair per KDA KV group. Pairs naming -1
 * raise LMC_ST_NO_BLOCK, ids outside [0, num_blocks) LMC_ST_BLOCK_OOR; such
 * pairs are skipped. The pairs of one call run concurrently, so the call
 * checks, on `host_pairs` and before anything is enqueued, that among the
 * pairs it will copy no block is the destination of two pairs or the
 * destination of one and the source of another, across all KV groups (a
 * block id names the same block in every group): LMC_ERR_OVERLAP otherwise,
 * and nothing is copied. The device pairs must equal the host pairs (the
 * kernels read the device copy). Asynchronous on `stream`; errors
 * INVALID_ARG (host_pairs missing), OVERLAP, ALIGN, CUDA. */
LMC_API int lmc_copy_blocks(const lmc_layout *layout, void *pool, const lmc_copy_batch *batch, uint32_t *status,
                    void *stream);

/* Guard for a mixed serving step ([HM] object groups; [VB] §5.3 a hit's state
 * becomes the initial state): a load of cached chunks and a store of new
 * chunks issued at the same time on one pool race unless they touch disjoint
 * blocks. Given two chunk-form batches whose block tables and jobs are in
 * HOST memory (the copies the caller built them from), computes the blocks
 * each one's objects read or write, exactly as lmc_store / lmc_load address
 * them: a paged layer's m = chunk_size / N positions of the chunk, a KDA
 * layer's chunk-end position. A job naming no request of its batch or a
 * negative chunk, a position past its table and an id outside the pool
 * touch nothing. Arena offsets are not looked at (there is no arena), so a
 * job the kernels would refuse for its offset still counts. Returns LMC_OK
 * when no block is touched by both, else LMC_ERR_OVERLAP with *out_block
 * (if not NULL) = the smallest shared block id (-1 when disjoint).
 * Errors: INVALID_ARG, NOT_MULTIPLE, OVERFLOW. Host only; nothing enqueued. */
LMC_API int lmc_check_disjoint(const lmc_layout *layout, int64_t chunk_size, const lmc_batch *a, const lmc_batch *b,
                               int32_t *out_block);

/* The same guard for block-granular batches (as lmc_store_blocks /
 * lmc_load_blocks address them): each job's object covers blocks_per_object
 * positions from its first block position, all of them for a paged layer,
 * and for a KDA layer the last one (LMC_KDA_LAST_BLOCK) or all of them
 * (LMC_KDA_EVERY_BLOCK). The INT8 forms address the same blocks. When the
 * two batches use different KDA modes, pass LMC_KDA_EVERY_BLOCK: it counts
 * a superset of the blocks either form touches. Results as
 * lmc_check_disjoint; errors INVALID_ARG. Host only; nothing enqueued. */
LMC_API int lmc_check_disjoint_blocks(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                                      const lmc_batch *a, const lmc_batch *b, int32_t *out_block);

/* ---- INT8 per-channel codec of the KDA recurrent state ------------------- */

/* Chunk-form store/load that keeps every KDA snapshot as an INT8 record
 * ([MC] "Compressed Checkpoint Storage": inactive recurrent states are
 * compressed to INT8 with per-channel parameters; the convolution window
 * keeps its original precision; a hit is decoded back to full precision).
 * The page is read as conv_state (conv_bytes, copied as is) followed by the
 * fp32 recurrent state in rows of `row_elems` values (heads * d rows of d for
 * a (heads, d, d) state). Per row: scale = max|x| / 127; code = x / scale
 * rounded half to even, clamped to [-127, 127]; an all-zero row has scale 0;
 * decoded value = code * scale; all IEEE binary32. A KDA layer's record in the
 * object: conv bytes, then one fp32 scale per row, then the int8 codes, row
 * by row. Paged layers are stored exactly as by lmc_store. Lossy: a decoded
 * value lies within half a step (scale / 2) of the original. States holding
 * NaN or infinity are outside the codec's domain (the output is unspecified).
 * Requires 4 <= row_elems <= 512, row_elems % 4 == 0, every KDA layer's
 * recurrent state a whole number of rows and a multiple of 4 rows, and
 * conv_bytes a multiple of 16, so records stay multiples of 16 bytes
 * (INVALID_ARG otherwise), and 16-byte aligned pool and arena (ALIGN).
 * Every layout of up to LMC_MAX_LAYERS layers fits one launch, KDA layers
 * included (their records take two launch-plan entries each). Other
 * arguments, status bits and errors as lmc_store / lmc_load. */
LMC_API int lmc_store_q8(const lmc_layout *layout, int64_t chunk_size, int64_t row_elems, const void *pool,
                 const lmc_batch *batch, void *arena, int64_t arena_bytes, uint32_t *status, void *stream);
LMC_API int lmc_load_q8(const lmc_layout *layout, int64_t chunk_size, int64_t row_elems, void *pool,
                const lmc_batch *batch, const void *arena, int64_t arena_bytes, uint32_t *status,
                void *stream);

/* Bytes of one chunk object of `object_group` as lmc_store_q8 writes it. */
LMC_API int lmc_object_bytes_q8(const lmc_layout *layout, int64_t chunk_size, int64_t row_elems, int32_t object_group,
                        int64_t *out);

/* Block-granular store/load (as lmc_store_blocks / lmc_load_blocks) with
 * every stored KDA snapshot kept as an INT8 record as lmc_store_q8 does: the
 * checkpoints taken at block boundaries ([KL] align mode) compressed for
 * storage ([MC] "Compressed Checkpoint Storage"). With LMC_KDA_EVERY_BLOCK a
 * KDA layer holds blocks_per_object records, one per block in order, each
 * conv bytes, scales, codes; with LMC_KDA_LAST_BLOCK one record, that of the
 * object's last block. Row rules, status bits and errors as lmc_store_q8. */
LMC_API int lmc_store_blocks_q8(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                                int64_t row_elems, const void *pool, const lmc_batch *batch, void *arena,
                                int64_t arena_bytes, uint32_t *status, void *stream);
LMC_API int lmc_load_blocks_q8(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                               int64_t row_elems, void *pool, const lmc_batch *batch, const void *arena,
                               int64_t arena_bytes, uint32_t *status, void *stream);

/* Bytes of one block-granular object of `object_group` as lmc_store_blocks_q8
 * writes it. */
LMC_API int lmc_object_bytes_blocks_q8(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                                       int64_t row_elems, int32_t object_group, int64_t *out);

/* ---- diagnostics ----------------------------------------------------------- */

/* Self-test of the device-side failure reporting: launches one thread that
 * polls, with the same bounded wait the bulk-copy engine uses, an mbarrier
 * that nothing completes, and ORs LMC_ST_TIMEOUT into *status (device)
 * after `rounds` polls (1 .. 2^22); no copy is in flight, so the context
 * stays usable. No counterpart on the pages (it tests this library's own
 * error path). Errors: INVALID_ARG, ALIGN, CUDA. */
LMC_API int lmc_selftest_wait(uint32_t *status, int64_t rounds, void *stream);

/* Self-test of the INT8 codec's row scale (see lmc_store_q8): for each of
 * the n fp32 values amax[i] (device, 4-byte aligned), writes the scale the
 * encoder stores (which must equal amax / 127 in IEEE binary32 division),
 * the inverse it multiplies by (0 where the encoder divides instead) and,
 * for comparison, the quotient by CUDA's IEEE division. Only finite,
 * non-negative amax is meaningful (a row maximum). No counterpart on the
 * pages (it tests this library's arithmetic). Errors: INVALID_ARG, ALIGN,
 * CUDA. */
LMC_API int lmc_selftest_row_scale(const float *amax, float *scale, float *inv, float *ieee, int64_t n,
                                   void *stream);

/* Static description of a code ("LMC_OK", ...); never NULL. */
LMC_API const char *lmc_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* LMC_H */

/*
 * oracle.c -- plain CPU oracle for paging a hybrid KDA + MLA model's cache
 * between a paged pool and per-chunk objects.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library. The product library never links,
 * includes or calls it, and it shares no code with the product.
 *
 * Apart from the INT8 codec of the KDA recurrent state (IEEE binary32
 * arithmetic, spelled out where it is defined), everything here is integer
 * arithmetic and memcpy, so "correct" means byte-identical.
 *
 * Sources (page title, section):
 *   [KL]  "Kimi-Linear" (LMCache recipe): chunk size a multiple of N; the
 *         [N, 2N) scheduler budget; snapshots at block boundaries.
 *   [K3]  "Kimi K3" (LMCache recipe): --chunk-size is a minimum, negotiated
 *         to the smallest multiple of N at or above it.
 *   [VB]  "How vLLM manages the KV cache of hybrid models: Kimi Linear /
 *         Kimi K3" (blog): §2.1 KDA state shapes, §2.2 grouping by equal
 *         spec, §3.1 padded shared-tensor layout (path A), §3.2 packed layout
 *         (path B), §4 the byte buffer and its per-layer views.
 *   [MC]  "When Prefix Cache Meets KDA" (Mooncake post), section "Flat KV":
 *         69 KDA layers split into three groups of 23, plus the
 *         full-attention group, on 24 physical slabs; "Copy-on-Write" /
 *         "Snapshot" (in-pool block copies); "Compressed Checkpoint Storage"
 *         (per-channel INT8 recurrent state, conv window kept).
 *   [HM]  "Hybrid Attention Models" (LMCache docs), "Object-group
 *         separation": one object group per cross-chunk attention window.
 *
 * Readings where the pages leave a step open (each is listed in the design
 * notes): equal-spec layers are split into near-equal runs whose count is
 * fixed by the smallest per-spec layer count; slab t holds the t-th layer of
 * every group; objects are layer-major in model order and token-major within
 * a paged layer; a KDA object holds the snapshot of the chunk's last block;
 * object offsets must be multiples of 16 bytes.
 *
 * Parity status: negotiation and layout sizes are pinned by values and
 * closed forms from the pages; store/load are pinned by invariants (identity,
 * untouched bytes) and by an independent per-token brute force; the codec by
 * worked rows and an independent float32 restatement; the rule refusing
 * racing block copies by the brute force applying each batch in several
 * orders; the mixed step's disjointness check by the brute force storing
 * each batch from a pool whose pages hold their block id. The byte order
 * inside an object is a reading, not a value from the pages.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

/* ------------------------------------------------------------------ */
/* Chunk-size negotiation ([K3] "Chunk-Size Negotiation"; [KL], [HM]    */
/* Step 2 for the strict form).                                         */
/* ------------------------------------------------------------------ */
int or_negotiate_chunk(int64_t requested, int64_t N, int strict, int64_t *out)
{
    if (out == NULL || N <= 0)
        return OR_ERR_INVALID_ARG;
    if (strict) {
        /* Strict form: the chunk must already be a positive multiple of N. */
        if (requested <= 0)
            return OR_ERR_INVALID_ARG;
        if (requested % N != 0)
            return OR_ERR_NOT_MULTIPLE;
        *out = requested;
        return OR_OK;
    }
    /* The least multiple of N not below `requested`; a minimum at or below
     * zero negotiates to N itself. */
    if (requested <= 0) {
        *out = N;
        return OR_OK;
    }
    int64_t k = requested / N;
    if (requested % N != 0)
        k += 1;
    if (k > INT64_MAX / N)
        return OR_ERR_OVERFLOW;
    *out = k * N;
    return OR_OK;
}

/* Scheduler budget rule ([KL] "Why these settings"; [HM] Step 2):
 * budget in [N, 2N) always; >= 2N only with separate object groups. */
int or_check_step_budget(int64_t N, int64_t max_batched, int separate_object_groups)
{
    if (N <= 0 || max_batched <= 0)
        return OR_ERR_INVALID_ARG;
    if (max_batched < N)
        return OR_ERR_BUDGET;
    if (max_batched < 2 * N)
        return OR_OK;
    return separate_object_groups ? OR_OK : OR_ERR_BUDGET;
}

/* Which backends can read a layout ([VB] §3.3): padding an attention
 * layer's page (padded path, its page smaller than the unified page) needs an
 * attention backend that indexes pages by the block stride; the packed path
 * needs every backend to address pages by the block stride, and KDA kernels
 * that assume contiguous pages cannot. Returns the OR_BK_* bits of every
 * rule the layout breaks (0: readable). */
uint32_t or_check_backends(const or_layout *L, int attn_indexes_by_stride, int state_pages_strided_ok)
{
    uint32_t bad = 0;
    for (int i = 0; i < L->num_layers; i++) {
        int attention = L->layers[i].kind != OR_KDA;
        if (!L->packed) {
            if (attention && L->page_bytes[i] > L->real_bytes[i] && !attn_indexes_by_stride)
                bad |= OR_BK_PADDED_ATTENTION;
        } else {
            if (attention && !attn_indexes_by_stride)
                bad |= OR_BK_PACKED_ATTENTION;
            if (!attention && !state_pages_strided_ok)
                bad |= OR_BK_PACKED_STATE;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Layout ([VB] §2.1, §2.2, §3.1, §3.2, §4; [MC] "Flat KV").            */
/* ------------------------------------------------------------------ */

/* Bytes of one layer's page that hold data. A paged attention layer keeps
 * one token_bytes entry per token of an N-token block ([VB] §4.2, view
 * (num_blocks, block_size, latent)). A KDA layer keeps conv_state plus
 * recurrent_state, independent of sequence length ([VB] §2.1). */
static int64_t real_page_bytes(const or_layer *l, int64_t N)
{
    if (l->kind == OR_KDA)
        return l->conv_bytes + l->rec_bytes;
    return N * l->token_bytes;
}

static int same_spec(const or_layer *a, const or_layer *b)
{
    return a->kind == b->kind && a->token_bytes == b->token_bytes &&
           a->conv_bytes == b->conv_bytes && a->rec_bytes == b->rec_bytes &&
           a->window == b->window;
}

/* Object-group class of a layer ([HM] "Object-group separation"): full
 * attention is one window; KDA (a mamba-like state) is another; each
 * sliding-window size is its own. */
static int same_window_class(const or_layer *a, const or_layer *b)
{
    if (a->kind != b->kind)
        return 0;
    if (a->kind == OR_SWA)
        return a->window == b->window;
    return 1;
}

int or_layout_build(or_layout *L)
{
    if (L == NULL)
        return OR_ERR_INVALID_ARG;
    int n = L->num_layers;
    if (n <= 0 || n > OR_MAX_LAYERS || L->N <= 0 || L->mem_bytes < 0)
        return OR_ERR_INVALID_ARG;
    for (int i = 0; i < n; i++) {
        const or_layer *l = &L->layers[i];
        if (l->kind == OR_KDA) {
            if (l->conv_bytes < 0 || l->rec_bytes < 0 || l->conv_bytes + l->rec_bytes <= 0)
                return OR_ERR_INVALID_ARG;
        } else if (l->kind == OR_MLA || l->kind == OR_SWA) {
            if (l->token_bytes <= 0)
                return OR_ERR_INVALID_ARG;
            if (l->kind == OR_SWA && l->window <= 0)
                return OR_ERR_INVALID_ARG;
            if (l->token_bytes > INT64_MAX / L->N)
                return OR_ERR_OVERFLOW;
        } else {
            return OR_ERR_INVALID_ARG;
        }
    }

    /* Step 1: bucket layers by equal spec, specs in order of first
     * appearance ([VB] §2.2: same_type_layers keyed by the spec). */
    int spec_of[OR_MAX_LAYERS];
    int spec_first[OR_MAX_LAYERS];
    int spec_count[OR_MAX_LAYERS];
    int num_specs = 0;
    for (int i = 0; i < n; i++) {
        int s;
        for (s = 0; s < num_specs; s++)
            if (same_spec(&L->layers[spec_first[s]], &L->layers[i]))
                break;
        if (s == num_specs) {
            spec_first[s] = i;
            spec_count[s] = 0;
            num_specs++;
        }
        spec_of[i] = s;
        spec_count[s]++;
    }

    /* Step 2: split each spec's layers into consecutive runs. With
     * split_groups set, the number of runs of a spec is
     * ceil(count / smallest count) and runs are near-equal, longer first;
     * for Kimi K3 this gives 3 KDA groups of 23 and one MLA group of 24,
     * i.e. 24 slabs ([MC] "Flat KV"). Otherwise one group per spec. */
    int smallest = spec_count[0];
    for (int s = 1; s < num_specs; s++)
        if (spec_count[s] < smallest)
            smallest = spec_count[s];
    int g = 0;
    int S = 0;
    for (int s = 0; s < num_specs; s++) {
        int cnt = spec_count[s];
        int runs = 1;
        if (L->split_groups)
            runs = (cnt + smallest - 1) / smallest;
        int base_len = cnt / runs;
        int extra = cnt % runs;
        int run = 0;
        int pos_in_run = 0;
        int run_len = base_len + (run < extra ? 1 : 0);
        for (int i = 0; i < n; i++) {
            if (spec_of[i] != s)
                continue;
            if (pos_in_run == run_len) {
                run++;
                pos_in_run = 0;
                run_len = base_len + (run < extra ? 1 : 0);
            }
            L->kv_group[i] = g + run;
            L->slot[i] = pos_in_run;
            pos_in_run++;
        }
        for (int r = 0; r < runs; r++) {
            int len = base_len + (r < extra ? 1 : 0);
            L->kv_group_kind[g + r] = L->layers[spec_first[s]].kind;
            L->kv_group_size[g + r] = len;
            if (len > S)
                S = len;
        }
        g += runs;
    }
    L->num_kv_groups = g;
    L->num_slabs = S;

    /* Step 3: object groups, one per cross-chunk window class in order of
     * first appearance, or a single group when separation is off. */
    int og_first[OR_MAX_LAYERS];
    int num_og = 0;
    for (int i = 0; i < n; i++) {
        if (!L->separate_object_groups) {
            L->object_group[i] = 0;
            num_og = 1;
            continue;
        }
        int o;
        for (o = 0; o < num_og; o++)
            if (same_window_class(&L->layers[og_first[o]], &L->layers[i]))
                break;
        if (o == num_og) {
            og_first[o] = i;
            num_og++;
        }
        L->object_group[i] = o;
    }
    L->num_object_groups = num_og;

    for (int i = 0; i < n; i++)
        L->real_bytes[i] = real_page_bytes(&L->layers[i], L->N);

    if (!L->packed) {
        /* Path A ([VB] §3.1): one page size for every layer, the largest
         * real page; smaller pages are padded up to it. Slab t is one tensor
         * of page_size * num_blocks bytes shared by the t-th layer of every
         * group, and block b sits at b * page_size inside it. */
        int64_t page = 0;
        for (int i = 0; i < n; i++)
            if (L->real_bytes[i] > page)
                page = L->real_bytes[i];
        if (page > INT64_MAX / S)
            return OR_ERR_OVERFLOW;
        int64_t per_block = page * (int64_t)S;
        int64_t nb = L->mem_bytes / per_block;
        if (nb <= 0)
            return OR_ERR_NO_MEMORY;
        L->page_size = page;
        L->block_stride = page;
        L->num_blocks = nb;
        L->pool_bytes = nb * per_block;
        for (int i = 0; i < n; i++) {
            L->page_bytes[i] = page;
            L->stride[i] = page;
            L->base[i] = (int64_t)L->slot[i] * page * nb;
        }
    } else {
        /* Path B ([VB] §3.2): within each group, byte offsets accumulate
         * over its layers' real pages; the block stride is the largest
         * group total; num_blocks = memory // block_stride; each layer is
         * the strided view (offset, block_stride) of one backing. */
        int64_t offset_in_group[OR_MAX_LAYERS];
        int64_t group_total[OR_MAX_LAYERS];
        for (int k = 0; k < L->num_kv_groups; k++)
            group_total[k] = 0;
        for (int k = 0; k < L->num_kv_groups; k++) {
            for (int t = 0; t < L->kv_group_size[k]; t++) {
                for (int i = 0; i < n; i++) {
                    if (L->kv_group[i] == k && L->slot[i] == t) {
                        offset_in_group[i] = group_total[k];
                        group_total[k] += L->real_bytes[i];
                    }
                }
            }
        }
        int64_t stride = 0;
        for (int k = 0; k < L->num_kv_groups; k++)
            if (group_total[k] > stride)
                stride = group_total[k];
        int64_t nb = L->mem_bytes / stride;
        if (nb <= 0)
            return OR_ERR_NO_MEMORY;
        L->page_size = 0;
        L->block_stride = stride;
        L->num_blocks = nb;
        L->pool_bytes = nb * stride;
        for (int i = 0; i < n; i++) {
            L->page_bytes[i] = L->real_bytes[i];
            L->stride[i] = stride;
            L->base[i] = offset_in_group[i];
        }
    }
    return OR_OK;
}

/* Bytes of one object of group og covering nb consecutive blocks: the
 * group's layers in model order; a paged layer holds all nb pages (the
 * object's tokens), a KDA layer one state snapshot (the last block's), or
 * nb snapshots (one per block) when kda_every is set. */
/* Bytes of a KDA page's INT8 record (codec below): conv bytes, one fp32
 * scale per row of d values, one int8 code per value. */
static int64_t q8_record_bytes(const or_layer *l, int64_t d)
{
    int64_t rows = l->rec_bytes / (4 * d);
    return l->conv_bytes + 4 * rows + rows * d;
}

static int64_t object_bytes_q(const or_layout *L, int64_t nb, int kda_every, int64_t q8_row, int og)
{
    int64_t total = 0;
    for (int i = 0; i < L->num_layers; i++) {
        if (L->object_group[i] != og)
            continue;
        int64_t page = L->real_bytes[i];
        if (L->layers[i].kind == OR_KDA && q8_row > 0)
            page = q8_record_bytes(&L->layers[i], q8_row);
        if (L->layers[i].kind == OR_KDA && !kda_every)
            total += page;
        else
            total += nb * page;
    }
    return total;
}

static int64_t object_bytes_nb(const or_layout *L, int64_t nb, int kda_every, int og)
{
    return object_bytes_q(L, nb, kda_every, 0, og);
}

/* Bytes of one object of group og for chunk size C (C / N blocks). */
int64_t or_object_bytes(const or_layout *L, int64_t C, int og)
{
    return object_bytes_nb(L, C / L->N, 0, og);
}

/* Bytes of one object of group og for a block-granular call. */
int64_t or_object_bytes_blocks(const or_layout *L, int64_t nb, int kda_every, int og)
{
    return object_bytes_nb(L, nb, kda_every, og);
}

/* ------------------------------------------------------------------ */
/* Store and load.                                                      */
/* ------------------------------------------------------------------ */

/* One page copy between the pool and an object, in either direction, or,
 * when `list` is given, a record of the page instead of the copy.
 * Returns the status bits raised (0 when the page was valid). */
static uint32_t copy_page(const or_layout *L, int layer, int64_t block,
                          uint8_t *pool, uint8_t *obj_bytes, int to_object,
                          uint32_t missing_bit, or_page_list *list, int64_t obj_offset)
{
    if (block == -1)
        return missing_bit;
    if (block < 0 || block >= L->num_blocks)
        return OR_ST_BLOCK_OOR;
    if (list != NULL) {
        if (list->count < list->capacity) {
            or_page *pg = &list->pages[list->count];
            pg->pool_offset = L->base[layer] + block * L->stride[layer];
            pg->object_offset = obj_offset;
            pg->bytes = L->real_bytes[layer];
            pg->layer = layer;
            pg->block = (int32_t)block;
        }
        list->count++;
        return 0;
    }
    uint8_t *page = pool + L->base[layer] + block * L->stride[layer];
    if (to_object)
        memcpy(obj_bytes, page, (size_t)L->real_bytes[layer]);
    else
        memcpy(page, obj_bytes, (size_t)L->real_bytes[layer]);
    return 0;
}

/* ------------------------------------------------------------------ */
/* INT8 per-channel codec of the KDA recurrent state ([MC] "Compressed  */
/* Checkpoint Storage": the recurrent state is quantised to INT8 with   */
/* per-channel parameters, the conv window kept in original precision). */
/* Readings: the page is conv_state then recurrent_state (fp32, rows of */
/* d values, row-major); a channel is one row; scale = max|x| / 127;    */
/* q = x / scale rounded half to even, clamped to [-127, 127]; an      */
/* all-zero row has scale 0 and codes 0; x' = q * scale. All in fp32.   */
/* Record of one page: conv bytes, then rows fp32 scales, then         */
/* rows * d int8 codes.                                                 */
/* ------------------------------------------------------------------ */

static void q8_encode(const uint8_t *page, uint8_t *rec, const or_layer *l, int64_t d)
{
    int64_t rows = l->rec_bytes / (4 * d);
    memcpy(rec, page, (size_t)l->conv_bytes);
    const uint8_t *x = page + l->conv_bytes;
    uint8_t *scales = rec + l->conv_bytes;
    int8_t *codes = (int8_t *)(rec + l->conv_bytes + 4 * rows);
    for (int64_t r = 0; r < rows; r++) {
        float amax = 0.0f;
        for (int64_t j = 0; j < d; j++) {
            float v;
            memcpy(&v, x + 4 * (r * d + j), 4);
            if (fabsf(v) > amax)
                amax = fabsf(v);
        }
        float scale = amax / 127.0f;
        memcpy(scales + 4 * r, &scale, 4);
        for (int64_t j = 0; j < d; j++) {
            float v;
            memcpy(&v, x + 4 * (r * d + j), 4);
            float q = 0.0f;
            if (scale != 0.0f) {
                q = rintf(v / scale);
                if (q > 127.0f)
                    q = 127.0f;
                if (q < -127.0f)
                    q = -127.0f;
            }
            codes[r * d + j] = (int8_t)q;
        }
    }
}

static void q8_decode(const uint8_t *rec, uint8_t *page, const or_layer *l, int64_t d)
{
    int64_t rows = l->rec_bytes / (4 * d);
    memcpy(page, rec, (size_t)l->conv_bytes);
    const uint8_t *scales = rec + l->conv_bytes;
    const int8_t *codes = (const int8_t *)(rec + l->conv_bytes + 4 * rows);
    uint8_t *x = page + l->conv_bytes;
    for (int64_t r = 0; r < rows; r++) {
        float scale;
        memcpy(&scale, scales + 4 * r, 4);
        for (int64_t j = 0; j < d; j++) {
            float v = (float)codes[r * d + j] * scale;
            memcpy(x + 4 * (r * d + j), &v, 4);
        }
    }
}

/* One KDA snapshot page <-> its compressed record (same checks as copy_page). */
static uint32_t q8_page(const or_layout *L, int layer, int64_t block, uint8_t *pool, uint8_t *rec,
                        int to_object, int64_t d, or_page_list *list, int64_t obj_offset)
{
    if (block == -1)
        return OR_ST_NO_SNAPSHOT;
    if (block < 0 || block >= L->num_blocks)
        return OR_ST_BLOCK_OOR;
    uint8_t *page = pool == NULL ? NULL : pool + L->base[layer] + block * L->stride[layer];
    if (list != NULL) {
        if (list->count < list->capacity) {
            or_page *pg = &list->pages[list->count];
            pg->pool_offset = L->base[layer] + block * L->stride[layer];
            pg->object_offset = obj_offset;
            pg->bytes = L->real_bytes[layer];
            pg->layer = layer;
            pg->block = (int32_t)block;
        }
        list->count++;
        return 0;
    }
    if (to_object)
        q8_encode(page, rec, &L->layers[layer], d);
    else
        q8_decode(rec, page, &L->layers[layer], d);
    return 0;
}

/* Row length d accepted by the codec: 4 <= d <= 512, d % 4 == 0, every KDA
 * layer's recurrent state a whole number of rows, a multiple of 4 rows, and
 * conv bytes a multiple of 16, so that every record (and every object) stays
 * a multiple of 16 bytes. */
static int q8_check(const or_layout *L, int64_t d)
{
    if (d < 4 || d > 512 || d % 4 != 0)
        return OR_ERR_INVALID_ARG;
    for (int i = 0; i < L->num_layers; i++)
        if (L->layers[i].kind == OR_KDA &&
            (L->layers[i].rec_bytes % (4 * d) != 0 || (L->layers[i].rec_bytes / (4 * d)) % 4 != 0 ||
             L->layers[i].conv_bytes % 16 != 0))
            return OR_ERR_INVALID_ARG;
    return OR_OK;
}

static int check_tables(const or_layout *L, const or_tables *T)
{
    if (T == NULL || T->num_kv_groups != L->num_kv_groups || T->num_requests < 0)
        return OR_ERR_INVALID_ARG;
    for (int k = 0; k < L->num_kv_groups; k++)
        if ((T->num_requests > 0 && T->table[k] == NULL) || T->num_cols[k] < 0 ||
            T->row_stride[k] < T->num_cols[k])
            return OR_ERR_INVALID_ARG;
    return OR_OK;
}

/* How the jobs of one call map to block positions: an object covers nb
 * consecutive positions starting at `first`, where first = chunk * nb for
 * chunk jobs and the job's own value for block jobs. */
typedef struct {
    int64_t nb;
    int first_is_block;
    int kda_every;
    int64_t q8_row; /* > 0: KDA snapshots as INT8 records with rows of q8_row values */
} obj_shape;

/* Moves every object of every job, in either direction. */
static int move_objects(const or_layout *L, const obj_shape *sh, uint8_t *pool,
                        const or_tables *T, const or_jobs *J,
                        uint8_t *arena, int64_t arena_bytes, uint32_t *status,
                        int to_object, or_page_list *list)
{
    if (L == NULL || (pool == NULL && list == NULL) || J == NULL || status == NULL)
        return OR_ERR_INVALID_ARG;
    int rc = check_tables(L, T);
    if (rc != OR_OK)
        return rc;
    if (J->num_object_groups != L->num_object_groups)
        return OR_ERR_INVALID_ARG;
    int64_t nb = sh->nb;

    for (int og = 0; og < L->num_object_groups; og++) {
        int64_t obj_size = object_bytes_q(L, nb, sh->kda_every, sh->q8_row, og);
        for (int64_t q = 0; q < J->num_jobs[og]; q++) {
            const or_job *job = &J->jobs[og][q];
            int64_t r = job->request;
            int64_t c = job->chunk;
            /* A job must name a request of the batch, a non-negative chunk,
             * and a 16-byte aligned object that fits the arena. */
            if (r < 0 || r >= T->num_requests || c < 0 || job->offset < 0 ||
                job->offset % 16 != 0 || obj_size > arena_bytes ||
                job->offset > arena_bytes - obj_size) {
                *status |= OR_ST_BAD_JOB;
                continue;
            }
            int64_t first = sh->first_is_block ? c : c * nb;
            uint8_t *obj = arena == NULL ? NULL : arena + job->offset;
            int64_t cursor = 0;
            for (int i = 0; i < L->num_layers; i++) {
                if (L->object_group[i] != og)
                    continue;
                int k = L->kv_group[i];
                const int32_t *row = T->table[k] + r * T->row_stride[k];
                if (L->layers[i].kind == OR_KDA && !sh->kda_every) {
                    /* The state a restore resumes from is the snapshot
                     * taken at the end of the object's last block ([KL]
                     * "Why these settings"; [MC] checkpoint boundaries). */
                    int64_t pos = first + nb - 1;
                    if (pos >= T->num_cols[k])
                        *status |= OR_ST_BAD_JOB;
                    else if (sh->q8_row > 0)
                        *status |= q8_page(L, i, row[pos], pool, obj + cursor, to_object,
                                           sh->q8_row, list, job->offset + cursor);
                    else
                        *status |= copy_page(L, i, row[pos], pool, obj + cursor,
                                             to_object, OR_ST_NO_SNAPSHOT, list,
                                             job->offset + cursor);
                    cursor += sh->q8_row > 0 ? q8_record_bytes(&L->layers[i], sh->q8_row)
                                             : L->real_bytes[i];
                } else if (L->layers[i].kind == OR_KDA) {
                    /* One snapshot per block boundary ([VB] §7, "all"-style
                     * snapshots kept per object). */
                    for (int64_t s = 0; s < nb; s++) {
                        int64_t pos = first + s;
                        if (pos >= T->num_cols[k])
                            *status |= OR_ST_BAD_JOB;
                        else if (sh->q8_row > 0)
                            *status |= q8_page(L, i, row[pos], pool, obj + cursor, to_object,
                                               sh->q8_row, list, job->offset + cursor);
                        else
                            *status |= copy_page(L, i, row[pos], pool, obj + cursor,
                                                 to_object, OR_ST_NO_SNAPSHOT, list,
                                                 job->offset + cursor);
                        cursor += sh->q8_row > 0 ? q8_record_bytes(&L->layers[i], sh->q8_row)
                                                 : L->real_bytes[i];
                    }
                } else {
                    /* The object's tokens are its nb consecutive blocks. */
                    for (int64_t j = 0; j < nb; j++) {
                        int64_t pos = first + j;
                        if (pos >= T->num_cols[k])
                            *status |= OR_ST_BAD_JOB;
                        else
                            *status |= copy_page(L, i, row[pos], pool, obj + cursor,
                                                 to_object, OR_ST_NO_BLOCK, list,
                                                 job->offset + cursor);
                        cursor += L->real_bytes[i];
                    }
                }
            }
        }
    }
    return OR_OK;
}

static int chunk_shape(const or_layout *L, int64_t C, obj_shape *sh)
{
    if (L == NULL)
        return OR_ERR_INVALID_ARG;
    if (C <= 0 || C % L->N != 0)
        return OR_ERR_NOT_MULTIPLE;
    sh->nb = C / L->N;
    sh->first_is_block = 0;
    sh->kda_every = 0;
    sh->q8_row = 0;
    return OR_OK;
}

static int block_shape(int64_t nb, int kda_every, obj_shape *sh)
{
    if (nb <= 0 || (kda_every != 0 && kda_every != 1))
        return OR_ERR_INVALID_ARG;
    sh->nb = nb;
    sh->first_is_block = 1;
    sh->kda_every = kda_every;
    sh->q8_row = 0;
    return OR_OK;
}

int or_store(const or_layout *L, int64_t C, const uint8_t *pool,
             const or_tables *T, const or_jobs *J,
             uint8_t *arena, int64_t arena_bytes, uint32_t *status)
{
    obj_shape sh;
    int rc = chunk_shape(L, C, &sh);
    if (rc != OR_OK)
        return rc;
    if (arena == NULL)
        return OR_ERR_INVALID_ARG;
    return move_objects(L, &sh, (uint8_t *)pool, T, J, arena, arena_bytes, status, 1, NULL);
}

int or_load(const or_layout *L, int64_t C, uint8_t *pool,
            const or_tables *T, const or_jobs *J,
            const uint8_t *arena, int64_t arena_bytes, uint32_t *status)
{
    obj_shape sh;
    int rc = chunk_shape(L, C, &sh);
    if (rc != OR_OK)
        return rc;
    if (arena == NULL)
        return OR_ERR_INVALID_ARG;
    return move_objects(L, &sh, pool, T, J, (uint8_t *)arena, arena_bytes, status, 0, NULL);
}

/* Block-granular store/load: every object covers nb consecutive block
 * positions from the job's own first position (its `chunk` field), e.g. the
 * whole blocks past a request's last whole chunk, or a chunk's blocks with
 * one KDA snapshot per block (kda_every). */
int or_store_blocks(const or_layout *L, int64_t nb, int kda_every, const uint8_t *pool,
                    const or_tables *T, const or_jobs *J,
                    uint8_t *arena, int64_t arena_bytes, uint32_t *status)
{
    obj_shape sh;
    int rc = block_shape(nb, kda_every, &sh);
    if (rc != OR_OK)
        return rc;
    if (arena == NULL)
        return OR_ERR_INVALID_ARG;
    return move_objects(L, &sh, (uint8_t *)pool, T, J, arena, arena_bytes, status, 1, NULL);
}

int or_load_blocks(const or_layout *L, int64_t nb, int kda_every, uint8_t *pool,
                   const or_tables *T, const or_jobs *J,
                   const uint8_t *arena, int64_t arena_bytes, uint32_t *status)
{
    obj_shape sh;
    int rc = block_shape(nb, kda_every, &sh);
    if (rc != OR_OK)
        return rc;
    if (arena == NULL)
        return OR_ERR_INVALID_ARG;
    return move_objects(L, &sh, pool, T, J, (uint8_t *)arena, arena_bytes, status, 0, NULL);
}

/* The pages a store or load of the jobs touches, in the order it touches
 * them, without moving bytes: pool offset, object offset (arena-relative)
 * and length of each. Used to check large cases one object at a time.
 * Returns OR_OK and sets list->count to the number of pages (records past
 * list->capacity are counted but not written). nb <= 0 selects the chunk
 * form with chunk size C; otherwise the block form. */
int or_list_pages_any(const or_layout *L, int64_t C, int64_t nb, int kda_every,
                      const or_tables *T, const or_jobs *J,
                      int64_t arena_bytes, uint32_t *status, or_page_list *list)
{
    if (list == NULL || (list->capacity > 0 && list->pages == NULL))
        return OR_ERR_INVALID_ARG;
    obj_shape sh;
    int rc = nb <= 0 ? chunk_shape(L, C, &sh) : block_shape(nb, kda_every, &sh);
    if (rc != OR_OK)
        return rc;
    list->count = 0;
    return move_objects(L, &sh, NULL, T, J, NULL, arena_bytes, status, 1, list);
}

int or_list_pages(const or_layout *L, int64_t C, const or_tables *T, const or_jobs *J,
                  int64_t arena_bytes, uint32_t *status, or_page_list *list)
{
    return or_list_pages_any(L, C, 0, 0, T, J, arena_bytes, status, list);
}

/* Chunk-form store/load with every KDA snapshot held as its INT8 record
 * (paged layers unchanged). d = values per recurrent-state row. */
int or_store_q8(const or_layout *L, int64_t C, int64_t d, const uint8_t *pool,
                const or_tables *T, const or_jobs *J,
                uint8_t *arena, int64_t arena_bytes, uint32_t *status)
{
    obj_shape sh;
    int rc = chunk_shape(L, C, &sh);
    if (rc == OR_OK)
        rc = q8_check(L, d);
    if (rc != OR_OK)
        return rc;
    if (arena == NULL)
        return OR_ERR_INVALID_ARG;
    sh.q8_row = d;
    return move_objects(L, &sh, (uint8_t *)pool, T, J, arena, arena_bytes, status, 1, NULL);
}

int or_load_q8(const or_layout *L, int64_t C, int64_t d, uint8_t *pool,
               const or_tables *T, const or_jobs *J,
               const uint8_t *arena, int64_t arena_bytes, uint32_t *status)
{
    obj_shape sh;
    int rc = chunk_shape(L, C, &sh);
    if (rc == OR_OK)
        rc = q8_check(L, d);
    if (rc != OR_OK)
        return rc;
    if (arena == NULL)
        return OR_ERR_INVALID_ARG;
    sh.q8_row = d;
    return move_objects(L, &sh, pool, T, J, (uint8_t *)arena, arena_bytes, status, 0, NULL);
}

/* Bytes of one chunk object of group og with compressed KDA records, or -1
 * when d is not accepted. */
int64_t or_object_bytes_q8(const or_layout *L, int64_t C, int64_t d, int og)
{
    if (q8_check(L, d) != OR_OK || C <= 0 || C % L->N != 0)
        return -1;
    return object_bytes_q(L, C / L->N, 0, d, og);
}

/* Block-granular store/load with every KDA snapshot (the last block's, or
 * one per block with kda_every) held as its INT8 record: the checkpoints of
 * [MC] "Compressed Checkpoint Storage" taken at block boundaries ([KL]). */
int or_store_blocks_q8(const or_layout *L, int64_t nb, int kda_every, int64_t d, const uint8_t *pool,
                       const or_tables *T, const or_jobs *J,
                       uint8_t *arena, int64_t arena_bytes, uint32_t *status)
{
    obj_shape sh;
    int rc = block_shape(nb, kda_every, &sh);
    if (rc == OR_OK)
        rc = q8_check(L, d);
    if (rc != OR_OK)
        return rc;
    if (arena == NULL)
        return OR_ERR_INVALID_ARG;
    sh.q8_row = d;
    return move_objects(L, &sh, (uint8_t *)pool, T, J, arena, arena_bytes, status, 1, NULL);
}

int or_load_blocks_q8(const or_layout *L, int64_t nb, int kda_every, int64_t d, uint8_t *pool,
                      const or_tables *T, const or_jobs *J,
                      const uint8_t *arena, int64_t arena_bytes, uint32_t *status)
{
    obj_shape sh;
    int rc = block_shape(nb, kda_every, &sh);
    if (rc == OR_OK)
        rc = q8_check(L, d);
    if (rc != OR_OK)
        return rc;
    if (arena == NULL)
        return OR_ERR_INVALID_ARG;
    sh.q8_row = d;
    return move_objects(L, &sh, pool, T, J, (uint8_t *)arena, arena_bytes, status, 0, NULL);
}

/* Bytes of one block-granular object of group og with INT8 KDA records, or
 * -1 when nb, kda_every or d is not accepted. */
int64_t or_object_bytes_blocks_q8(const or_layout *L, int64_t nb, int kda_every, int64_t d, int og)
{
    if (q8_check(L, d) != OR_OK || nb <= 0 || (kda_every != 0 && kda_every != 1))
        return -1;
    return object_bytes_q(L, nb, kda_every, d, og);
}

/* In-pool block copies ([MC] "Copy-on-Write", "Snapshot": a shared
 * checkpoint's state is copied into a private slot, a running state into a
 * spare buffer). For every pair of KV group g, each layer of g gets the real
 * bytes of block src copied to block dst. A pair naming -1 or a block outside
 * the pool is skipped and raises its bit. */
static int block_in_pool(const or_layout *L, int64_t b)
{
    return b >= 0 && b < L->num_blocks;
}

/* The pairs of one copy call are applied together, not one after another
 * ([MC] "Copy-on-Write": each hit gets its own private slot; "Snapshot":
 * each running state its own spare buffer), so a call is well defined only
 * if no block it writes is written again or read by another of its pairs.
 * A block id names one block for every KV group (the groups' pages of block
 * b share memory in both layouts), so pairs of different groups are
 * compared too. Pairs with an id outside the pool copy nothing and take no
 * part. Returns 1 when two pairs collide. */
static int copies_collide(const or_layout *L, const or_copy_batch *B)
{
    for (int g = 0; g < L->num_kv_groups; g++) {
        for (int64_t q = 0; q < B->num_pairs[g]; q++) {
            const or_pair *p = &B->pairs[g][q];
            if (!block_in_pool(L, p->src_block) || !block_in_pool(L, p->dst_block))
                continue;
            for (int h = 0; h < L->num_kv_groups; h++) {
                for (int64_t t = 0; t < B->num_pairs[h]; t++) {
                    const or_pair *o = &B->pairs[h][t];
                    if ((h == g && t == q) || !block_in_pool(L, o->src_block) ||
                        !block_in_pool(L, o->dst_block))
                        continue;
                    if (p->dst_block == o->dst_block || p->dst_block == o->src_block)
                        return 1;
                }
            }
        }
    }
    return 0;
}

int or_copy_blocks(const or_layout *L, uint8_t *pool, const or_copy_batch *B, uint32_t *status)
{
    if (L == NULL || pool == NULL || B == NULL || status == NULL ||
        B->num_kv_groups != L->num_kv_groups)
        return OR_ERR_INVALID_ARG;
    for (int g = 0; g < L->num_kv_groups; g++) {
        if (B->num_pairs[g] < 0 || (B->num_pairs[g] > 0 && B->pairs[g] == NULL))
            return OR_ERR_INVALID_ARG;
    }
    if (copies_collide(L, B))
        return OR_ERR_OVERLAP;
    for (int g = 0; g < L->num_kv_groups; g++) {
        for (int64_t q = 0; q < B->num_pairs[g]; q++) {
            int64_t src = B->pairs[g][q].src_block;
            int64_t dst = B->pairs[g][q].dst_block;
            if (src == -1 || dst == -1) {
                *status |= OR_ST_NO_BLOCK;
                continue;
            }
            if (src < 0 || src >= L->num_blocks || dst < 0 || dst >= L->num_blocks) {
                *status |= OR_ST_BLOCK_OOR;
                continue;
            }
            for (int i = 0; i < L->num_layers; i++) {
                if (L->kv_group[i] != g)
                    continue;
                memmove(pool + L->base[i] + dst * L->stride[i],
                        pool + L->base[i] + src * L->stride[i], (size_t)L->real_bytes[i]);
            }
        }
    }
    return OR_OK;
}

/* Sets `bit` in map[b] for every block b whose pages the objects of a
 * batch read (store) or write (load). An object covers nb block positions
 * from `first` (chunk jobs: chunk * nb; block jobs: the job's own value):
 * all of them for a paged layer; for a KDA layer the last one, the state at
 * the object's end ([KL] snapshots at block boundaries), or all of them
 * with kda_every. A job naming no request of the batch or a negative chunk,
 * a position past the table, and an id outside the pool mark nothing. */
static int mark_blocks(const or_layout *L, const obj_shape *sh, const or_tables *T, const or_jobs *J,
                       uint8_t *map, uint8_t bit)
{
    int rc = check_tables(L, T);
    if (rc != OR_OK)
        return rc;
    if (J == NULL || J->num_object_groups != L->num_object_groups)
        return OR_ERR_INVALID_ARG;
    for (int og = 0; og < L->num_object_groups; og++) {
        if (J->num_jobs[og] < 0 || (J->num_jobs[og] > 0 && J->jobs[og] == NULL))
            return OR_ERR_INVALID_ARG;
        for (int64_t q = 0; q < J->num_jobs[og]; q++) {
            int64_t r = J->jobs[og][q].request;
            int64_t c = J->jobs[og][q].chunk;
            if (r < 0 || r >= T->num_requests || c < 0)
                continue;
            for (int i = 0; i < L->num_layers; i++) {
                if (L->object_group[i] != og)
                    continue;
                int k = L->kv_group[i];
                int64_t first = sh->first_is_block ? c : c * sh->nb;
                int64_t lo = first, hi = first + sh->nb; /* positions [lo, hi) */
                if (L->layers[i].kind == OR_KDA && !sh->kda_every)
                    lo = hi - 1;
                for (int64_t pos = lo; pos < hi && pos < T->num_cols[k]; pos++) {
                    int64_t b = T->table[k][r * T->row_stride[k] + pos];
                    if (block_in_pool(L, b))
                        map[b] |= bit;
                }
            }
        }
    }
    return OR_OK;
}

/* A load and a store issued at the same time on one pool (the mixed
 * serving step) must touch disjoint blocks. *out_block = the smallest block
 * both touch, or -1. */
static int disjoint(const or_layout *L, const obj_shape *sh, const or_tables *Ta, const or_jobs *Ja,
                    const or_tables *Tb, const or_jobs *Jb, int32_t *out_block)
{
    uint8_t *map = calloc((size_t)L->num_blocks + 1, 1);
    if (map == NULL)
        return OR_ERR_INVALID_ARG;
    int rc = mark_blocks(L, sh, Ta, Ja, map, 1);
    if (rc == OR_OK)
        rc = mark_blocks(L, sh, Tb, Jb, map, 2);
    *out_block = -1;
    if (rc == OR_OK) {
        for (int64_t b = 0; b < L->num_blocks; b++) {
            if (map[b] == 3) {
                *out_block = (int32_t)b;
                rc = OR_ERR_OVERLAP;
                break;
            }
        }
    }
    free(map);
    return rc;
}

int or_check_disjoint(const or_layout *L, int64_t C, const or_tables *Ta, const or_jobs *Ja,
                      const or_tables *Tb, const or_jobs *Jb, int32_t *out_block)
{
    if (L == NULL || out_block == NULL)
        return OR_ERR_INVALID_ARG;
    obj_shape sh;
    int rc = chunk_shape(L, C, &sh);
    return rc != OR_OK ? rc : disjoint(L, &sh, Ta, Ja, Tb, Jb, out_block);
}

int or_check_disjoint_blocks(const or_layout *L, int64_t nb, int kda_every, const or_tables *Ta,
                             const or_jobs *Ja, const or_tables *Tb, const or_jobs *Jb, int32_t *out_block)
{
    if (L == NULL || out_block == NULL)
        return OR_ERR_INVALID_ARG;
    obj_shape sh;
    int rc = block_shape(nb, kda_every, &sh);
    return rc != OR_OK ? rc : disjoint(L, &sh, Ta, Ja, Tb, Jb, out_block);
}

/* Smallest multiple of `align` tokens whose attention page
 * (N * attn_token_bytes) holds at least state_page_bytes ([HM] Step 1: one
 * block size for all groups, large enough that the attention page is >= the
 * state page; [KL] note: 944 at TP 2 and 1888 at TP 1). Found by counting
 * up, one alignment step at a time. */
int or_unified_block_size(int64_t attn_token_bytes, int64_t state_page_bytes,
                          int64_t align, int64_t *out)
{
    if (out == NULL || attn_token_bytes <= 0 || state_page_bytes <= 0 || align <= 0)
        return OR_ERR_INVALID_ARG;
    int64_t n = align;
    while (n * attn_token_bytes < state_page_bytes) {
        if (n > INT64_MAX / attn_token_bytes - align)
            return OR_ERR_OVERFLOW;
        n += align;
    }
    *out = n;
    return OR_OK;
}

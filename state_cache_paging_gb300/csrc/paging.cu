// paging.cu -- store (gather pages -> chunk objects), load (scatter chunk
// objects -> pages), their INT8-codec forms for the KDA recurrent state, and
// in-pool block copies, for sm_103a.
//
// What is moved ("Hybrid Attention Models" (LMCache docs), Object-group
// separation; "Kimi-Linear" (LMCache recipe), Why these settings; "How vLLM
// manages the KV cache of hybrid models", §3.1/§3.2/§4/§7; "When Prefix Cache
// Meets KDA", Copy-on-Write / Snapshot): one object per (request, chunk or
// block range, object group); inside it, the group's layers in model order; a
// paged attention layer contributes the object's blocks, token-major, a KDA
// layer the state snapshot stored at the object's last block (or one per
// block). A block copy moves every layer page of one KV group from a source
// block to a destination block of the same pool. Every page is handled as
// opaque bytes: store, load and copy only move data, each byte read once from
// HBM and written once (the codec forms also touch each byte once, turning
// the KDA state rows into INT8 records and back).
//
// GPU design. The work of one launch is a flat list of tiles (each at most
// kTileBytes, 16-byte multiples, never crossing a page). Tile t resolves to
// (group, job, layer, page, piece) with integer math on the launch plan held
// in kernel parameter space, reads one block id (or one block pair) from the
// caller's device arrays, and copies one contiguous range: 32-byte (or, for
// ranges that are only 16-byte aligned, 16-byte) vector loads that bypass L1
// and streaming (evict-first) stores, several in flight per thread. One CTA
// per tile, several CTAs resident per SM, so the dependent block-table read
// of one CTA hides under the copies of others.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "lmc_internal.h"

// Defaults picked by measurement on GB300 (Kimi-Linear and K3 workloads):
// 32 KB tiles, 256 threads, four 32-byte vectors in flight per thread, i.e.
// one CTA moves its whole tile with a single round of loads and stores.
#ifndef LMC_TILE_BYTES
#define LMC_TILE_BYTES 32768
#endif
#ifndef LMC_THREADS
#define LMC_THREADS 256
#endif
#ifndef LMC_UNROLL
#define LMC_UNROLL 4
#endif
#ifndef LMC_MIN_BLOCKS
#define LMC_MIN_BLOCKS 1  // resident CTAs per SM the copy kernels are compiled for
#endif
#ifndef LMC_ENGINE
#define LMC_ENGINE 0  // 0: vector loads/stores, 1: bulk (TMA) copies through shared memory
#endif
#ifndef LMC_BULK_STAGES
#define LMC_BULK_STAGES 4
#endif
#ifndef LMC_BULK_CTAS_PER_SM
#define LMC_BULK_CTAS_PER_SM 1
#endif
#ifndef LMC_LD_HINT
#define LMC_LD_HINT 0  // 0: .nc.L1::no_allocate, 1: + .L2::256B prefetch, 2: plain
#endif
#ifndef LMC_ST_HINT
#define LMC_ST_HINT 0  // 0: .cs (evict-first), 1: plain write-back, 2: .L1::no_allocate
#endif

namespace {

constexpr int kMaxEntries = 2 * LMC_MAX_LAYERS;  // layer entries in one launch (a codec KDA layer takes two)
constexpr int kMaxGroups = 64;               // object groups (or KV groups) in one launch
constexpr int kMaxKv = 64;                   // KV groups (block tables)
constexpr int kTileBytes = LMC_TILE_BYTES;
constexpr int kThreads = LMC_THREADS;
constexpr int kUnroll = LMC_UNROLL;
constexpr int kEngine = LMC_ENGINE;
constexpr int kBulkStages = LMC_BULK_STAGES;
constexpr int kBulkCtasPerSm = LMC_BULK_CTAS_PER_SM;
static_assert(kEngine != 1 || kBulkCtasPerSm * (kBulkStages * kTileBytes + 1024) <= 228 * 1024,
              "bulk stages must fit the SM's shared memory");

enum Mode : int32_t { kStore = 0, kLoad = 1, kCopy = 2 };

// One layer's run of pages inside an object (or inside a copied block).
// A codec entry (INT8 record of a KDA recurrent state) counts rows instead
// of bytes: seg_bytes holds the page's state rows, tile_bytes the rows per
// tile, and pool_base points past the conv bytes, at the state itself.
struct Entry {
    int64_t pool_base;    // pool byte offset of block 0's page
    int64_t pool_stride;  // bytes between consecutive blocks' pages
    int64_t obj_off;      // byte offset of the layer's first page in the object
    int32_t seg_bytes;    // real bytes of one page
    int32_t tile_bytes;   // bytes per tile of this page (last tile shorter)
    int32_t tiles_per_seg;
    int32_t tile_start;   // tiles of earlier layers in the object
    int32_t obj_stride;   // bytes between the object's consecutive pages of this entry
    uint8_t kv;           // KV group (block table)
    uint8_t kda;          // 1: a KDA state page (a missing one is NO_SNAPSHOT)
    uint8_t codec;        // 1: INT8 record of the recurrent state (see below)
    uint8_t last;         // 1: only the object's last block position (block position =
                          // first + Plan::last_pos + page index; else first + page index)
};
static_assert(sizeof(Entry) == 48, "launch plan entry layout");
static_assert(kMaxKv <= 256, "KV group index held in one byte");

struct Group {
    const void *items;   // lmc_job[] (store/load) or lmc_block_pair[] (copy)
    int64_t num_items;
    int64_t tile_begin;  // first launch-wide tile of this group
    int64_t obj_bytes;
    int32_t tiles_per_obj;
    int32_t first_entry;
    int32_t num_entries;
    int32_t pad;
};

struct Table {
    const int32_t *ptr;
    int64_t row_stride;
    int64_t num_cols;
};

struct Plan {
    const uint8_t *src_base;  // store: pool; load: arena; copy: pool
    uint8_t *dst_base;        // store: arena; load: pool; copy: pool
    uint32_t *status;
    int64_t arena_bytes;
    int64_t num_blocks;
    int64_t total_tiles;
    int32_t pos_mul;  // first block position = job.chunk * pos_mul (C/N for chunk jobs, 1 for block jobs)
    int32_t num_requests;
    int32_t num_groups;
    int32_t mode;
    int32_t q8_row;    // codec: values per recurrent-state row (0: no codec)
    int32_t last_pos;  // block positions per object - 1 (the `last` entries' position offset)
    Group groups[kMaxGroups];
    Table tables[kMaxKv];
    Entry entries[kMaxEntries];
};
static_assert(sizeof(Plan) <= 32000, "kernel parameter space");

// Source bytes are read once: bypass L1 (and never alias the destination).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
#if LMC_LD_HINT == 0
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
#elif LMC_LD_HINT == 1
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
#else
    asm("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
#endif
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Destination bytes are not read back by this kernel.
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) {
#if LMC_ST_HINT == 0
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
#elif LMC_ST_HINT == 1
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
#else
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};"
#endif
                 ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// 32-byte (256-bit) loads and stores for tiles whose ends are 32-byte
// aligned, four in flight per thread (measured on GB300: +0-1.5 % over
// 16-byte vectors); other tiles take the 16-byte path.
#ifndef LMC_VEC32
#define LMC_VEC32 1
#endif
#ifndef LMC_VEC32_UNROLL
#define LMC_VEC32_UNROLL 4
#endif

struct alignas(32) u8x32 {
    uint4 lo, hi;
};

__device__ __forceinline__ u8x32 ld_stream32(const u8x32 *p) {
    u8x32 v;
    asm("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(v.lo.x), "=r"(v.lo.y), "=r"(v.lo.z), "=r"(v.lo.w), "=r"(v.hi.x), "=r"(v.hi.y), "=r"(v.hi.z),
          "=r"(v.hi.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream32(u8x32 *p, const u8x32 &v) {
    asm volatile("st.global.cs.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.lo.x), "r"(v.lo.y),
                 "r"(v.lo.z), "r"(v.lo.w), "r"(v.hi.x), "r"(v.hi.y), "r"(v.hi.z), "r"(v.hi.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// A resolved tile: copy `bytes` from src to dst.
struct Span {
    const uint8_t *src;
    uint8_t *dst;
    int32_t bytes;   // plain copy: bytes; codec: rows
    int32_t codec;   // 0: plain copy, 1: encode (store), 2: decode (load)
    uint8_t *scales; // codec: the rows' fp32 scales (written on encode, read on decode)
};

// Resolves tile -> span; returns the status bits to raise (0: copy it).
// kCodec compiles in the codec entries (only the INT8 kernels carry them).
template <bool kCodec>
__device__ __forceinline__ uint32_t resolve(const Plan &P, int64_t tile, Span &s) {
    // group: the last one whose first tile is <= tile
    int g = 0, gh = P.num_groups - 1;
    while (g < gh) {
        const int mid = (g + gh + 1) >> 1;
        if (P.groups[mid].tile_begin <= tile)
            g = mid;
        else
            gh = mid - 1;
    }
    const Group &G = P.groups[g];
    const int64_t local = tile - G.tile_begin;
    // job (or pair) index; a 32-bit division whenever the offset fits
    const int64_t q = local <= INT32_MAX ? (int64_t)((uint32_t)local / (uint32_t)G.tiles_per_obj)
                                         : local / G.tiles_per_obj;
    const int32_t t = (int32_t)(local - q * G.tiles_per_obj);

    // layer entry: the last one whose first tile is <= t
    int lo = G.first_entry, hi = G.first_entry + G.num_entries - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.entries[mid].tile_start <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    const Entry &E = P.entries[lo];
    const int32_t u = t - E.tile_start;
    const int32_t j = u / E.tiles_per_seg;  // page index within the layer
    const int32_t k = u - j * E.tiles_per_seg;
    const int64_t piece = (int64_t)k * E.tile_bytes;
    s.bytes = min(E.tile_bytes, (int32_t)(E.seg_bytes - piece));
    s.codec = 0;
    s.scales = nullptr;

    if (P.mode == kCopy) {
        const lmc_block_pair pr = static_cast<const lmc_block_pair *>(G.items)[q];
        if (pr.src_block == -1 || pr.dst_block == -1)
            return LMC_ST_NO_BLOCK;
        if (pr.src_block < 0 || pr.src_block >= P.num_blocks || pr.dst_block < 0 ||
            pr.dst_block >= P.num_blocks)
            return LMC_ST_BLOCK_OOR;
        s.src = P.src_base + E.pool_base + (int64_t)pr.src_block * E.pool_stride + piece;
        s.dst = P.dst_base + E.pool_base + (int64_t)pr.dst_block * E.pool_stride + piece;
        return 0;
    }

    const lmc_job job = static_cast<const lmc_job *>(G.items)[q];
    if (job.request < 0 || job.request >= P.num_requests || job.chunk < 0 || job.offset < 0 ||
        (job.offset & 15) != 0 || job.offset > P.arena_bytes - G.obj_bytes)
        return LMC_ST_BAD_JOB;
    const Table &T = P.tables[E.kv];
    const int64_t pos = (int64_t)job.chunk * P.pos_mul + (E.last ? P.last_pos : 0) + j;
    if (pos >= T.num_cols)
        return LMC_ST_BAD_JOB;
    const int32_t block = __ldg(T.ptr + (int64_t)job.request * T.row_stride + pos);
    if (block == -1)
        return E.kda ? LMC_ST_NO_SNAPSHOT : LMC_ST_NO_BLOCK;
    if (block < 0 || block >= P.num_blocks)
        return LMC_ST_BLOCK_OOR;

    if (kCodec && E.codec) {
        // rows [row0, row0 + s.bytes) of the page's recurrent state (pool_base
        // already points past the conv bytes; seg_bytes counts the rows); the
        // entry's j-th record part, at obj_off + j * obj_stride, holds all the
        // rows' scales, then the codes
        const int64_t row0 = piece;
        const int64_t page = E.pool_base + (int64_t)block * E.pool_stride + row0 * 4 * P.q8_row;
        const int64_t rec = job.offset + E.obj_off + (int64_t)j * E.obj_stride;
        const int64_t codes = rec + 4 * (int64_t)E.seg_bytes + row0 * P.q8_row;
        if (P.mode == kStore) {
            s.codec = 1;
            s.src = P.src_base + page;
            s.dst = P.dst_base + codes;
            s.scales = P.dst_base + rec + 4 * row0;
        } else {
            s.codec = 2;
            s.src = P.src_base + codes;
            s.dst = P.dst_base + page;
            s.scales = const_cast<uint8_t *>(P.src_base) + rec + 4 * row0;
        }
        return 0;
    }
    const int64_t page = E.pool_base + (int64_t)block * E.pool_stride + piece;
    const int64_t obj = job.offset + E.obj_off + (int64_t)j * E.obj_stride + piece;
    s.src = P.src_base + (P.mode == kStore ? page : obj);
    s.dst = P.dst_base + (P.mode == kStore ? obj : page);
    return 0;
}

// INT8 per-channel codec of the KDA recurrent state ("When Prefix Cache
// Meets KDA", Compressed Checkpoint Storage): per row of d fp32 values,
// scale = max|x| / 127, code = x / scale rounded half to even and clamped to
// [-127, 127] (IEEE binary32 division), zero rows give scale 0 and codes 0;
// decode = code * scale.
//
// Encode work split: a row's d / 4 float4 vectors are spread over `lpr` lanes
// of a warp, kRowVec consecutive vectors per lane, so 32 / lpr rows share a
// warp; the row maximum is a shuffle reduction inside each aligned group of
// lpr lanes. Each thread stages its vectors of the next kQ8Stages - 1 rounds
// in shared memory with asynchronous copies (cp.async: no registers held, and
// each thread waits only on its own copy groups), so loads stay in flight
// during the arithmetic.
// This needs d % (4 * kRowVec) == 0 and lpr = d / (4 * kRowVec) a power of two
// <= 32 (two float4 per lane: d = 8 .. 256 in powers of two); other row
// lengths take one row per warp. Decode is flat over the tile's codes: 16
// codes (one 16-byte load) per thread per round, kDecUnroll rounds of loads
// issued before their stores, values written as whole 32-byte sectors.
// Codec kernel shapes picked by measurement on GB300 (Kimi-Linear, d = 128):
// encoder 128 threads x 10 CTAs, four stages (three rounds ahead, 16 KB of
// shared memory per CTA): 7.10 TB/s (3 stages 7.00, 5 stages 7.03, 11 CTAs
// 6.94, 9 CTAs 6.99; 256-thread CTAs 5.9 since a 64-row tile then runs only
// two rounds; the next round prefetched in registers instead: 6.70 at
// 128 x 12; preferring the largest shared-memory carveout cost up to 3 %, so
// the driver's default split is kept); decoder 256 x 6 with two rounds in
// flight (7.02 TB/s).
#ifndef LMC_ROW_VEC
#define LMC_ROW_VEC 2
#endif
#ifndef LMC_Q8_ENC_THREADS
#define LMC_Q8_ENC_THREADS 128
#endif
#ifndef LMC_Q8_ENC_MIN_BLOCKS
#define LMC_Q8_ENC_MIN_BLOCKS 10
#endif
#ifndef LMC_Q8_DEC_THREADS
#define LMC_Q8_DEC_THREADS 256
#endif
#ifndef LMC_Q8_DEC_MIN_BLOCKS
#define LMC_Q8_DEC_MIN_BLOCKS 6
#endif
#ifndef LMC_Q8_DEC_UNROLL
#define LMC_Q8_DEC_UNROLL 2
#endif
#ifndef LMC_Q8_COPY_UNROLL
#define LMC_Q8_COPY_UNROLL 1  // vectors per thread per round on the codec kernels' plain pages
#endif
#ifndef LMC_Q8_STAGES
#define LMC_Q8_STAGES 4  // encoder: rounds staged in shared memory (kQ8Stages - 1 ahead)
#endif
#ifndef LMC_Q8_TILE_BYTES
#define LMC_Q8_TILE_BYTES 32768  // fp32 state bytes per codec tile
#endif
constexpr int kRowVec = LMC_ROW_VEC;
constexpr int kQ8TileBytes = LMC_Q8_TILE_BYTES;
constexpr int kDecUnroll = LMC_Q8_DEC_UNROLL;
constexpr int kQ8Stages = LMC_Q8_STAGES;
static_assert(kQ8Stages >= 2, "the staged encoder needs at least two stages");

// Rounding by addition: for |y| <= 2^22, RN(y + 1.5 * 2^23) equals
// 1.5 * 2^23 + rint(y) (ties to even: the floats of [2^23, 2^24) are the
// integers, and 1.5 * 2^23 is even), and since the bit pattern of 1.5 * 2^23
// ends in a zero byte, the low byte of the sum's bit pattern is rint(y) as a
// two's-complement byte.
constexpr float kRoundAdd = 12582912.0f;  // 1.5 * 2^23

struct RowScale {
    float scale;  // RN(max|x| / 127)
    float inv;    // ~1 / scale (relative error <= 2^-22), 0 for a zero row
    bool exact;   // tiny or huge maximum: every code by the IEEE quotient
};

// scale = RN(amax / 127) by Markstein's correction of a reciprocal product
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(amax * z)
// with z = RN(1 / 127) is within an ulp of the quotient, the residual
// r = amax - 127 * q0 is exact with one FMA, and RN(q0 + r * z) is the
// correctly rounded quotient (checked against the IEEE division for every
// finite non-negative amax). Below 2^-100 (subnormal quotients) the IEEE
// division itself is used. inv = RN(127 * rcp.approx(amax)): within 2^-22
// of 1 / scale, so |x * inv - x / scale| <= 127 * 2^-22 < 4e-5 for |x| <= amax.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ RowScale row_scale(float amax) {
    constexpr float kInv127 = 1.0f / 127.0f;
    RowScale rs;
    if (amax >= 7.88860905e-31f) {  // 2^-100
        const float q0 = amax * kInv127;
        rs.scale = fmaf(fmaf(-q0, 127.0f, amax), kInv127, q0);
    } else {
        rs.scale = __fdiv_rn(amax, 127.0f);
    }
    rs.exact = amax != 0.0f && (amax < 7.88860905e-31f || amax > 4.25352959e37f);  // outside [2^-100, 2^125]
    rs.inv = (amax == 0.0f || rs.exact) ? 0.0f : 127.0f * rcp_approx(amax);
    return rs;
}

// Maximum over each aligned group of `lanes` lanes (a power of two), by a
// butterfly of shuffles (measured faster here than redux.sync on the bit
// patterns).
__device__ __forceinline__ float group_max(float v, int lanes) {
    for (int o = lanes >> 1; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ uint32_t pack_low_bytes(float t0, float t1, float t2, float t3) {
    const uint32_t lo = __byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x0040);
    const uint32_t hi = __byte_perm(__float_as_uint(t2), __float_as_uint(t3), 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

// Four codes, packed little-endian: t = RN(x * inv + 1.5 * 2^23) rounds the
// exact product x * inv, which lies within 4e-5 of the exact quotient
// x / scale, and RN(x / scale) lies within 8e-6 of it. So unless the product
// is within 1e-4 of a half-integer, rint(RN(x / scale)) equals the product's
// rounding; `worst` collects |x * inv - rint| (one rounding of an exact
// residual) so the caller can tell. For a zero row (inv = 0) every code is 0;
// |x * inv| < 127.01 keeps every code inside [-127, 127].
__device__ __forceinline__ uint32_t quant4(const float4 &v, float inv, float &worst) {
    const float t0 = fmaf(v.x, inv, kRoundAdd), t1 = fmaf(v.y, inv, kRoundAdd);
    const float t2 = fmaf(v.z, inv, kRoundAdd), t3 = fmaf(v.w, inv, kRoundAdd);
    const float e0 = fmaf(v.x, inv, kRoundAdd - t0), e1 = fmaf(v.y, inv, kRoundAdd - t1);
    const float e2 = fmaf(v.z, inv, kRoundAdd - t2), e3 = fmaf(v.w, inv, kRoundAdd - t3);
    worst = fmaxf(worst, fmaxf(fmaxf(fabsf(e0), fabsf(e1)), fmaxf(fabsf(e2), fabsf(e3))));
    return pack_low_bytes(t0, t1, t2, t3);
}

// The same four codes by the definition: IEEE quotient, rint, clamp.
__device__ __forceinline__ uint32_t quant4_exact(const float4 &v, float scale) {
    if (scale == 0.0f)
        return 0u;
    const float c[4] = {v.x, v.y, v.z, v.w};
    float t[4];
#pragma unroll
    for (int k = 0; k < 4; k++)
        t[k] = fminf(127.0f, fmaxf(-127.0f, rintf(__fdiv_rn(c[k], scale)))) + kRoundAdd;
    return pack_low_bytes(t[0], t[1], t[2], t[3]);
}

// A lane's share of a row: if any product came within 1e-4 of a half-integer
// (or the row's maximum is tiny or huge) every code is recomputed by the
// definition.
template <int kN>
__device__ __forceinline__ void quant_lane(const float4 (&v)[kN], const RowScale &rs, uint32_t (&q)[kN]) {
    float worst = 0.0f;
#pragma unroll
    for (int w = 0; w < kN; w++)
        q[w] = quant4(v[w], rs.inv, worst);
    if (rs.exact || worst > 0.4999f) {
#pragma unroll
        for (int w = 0; w < kN; w++)
            q[w] = quant4_exact(v[w], rs.scale);
    }
}

// Four values from four codes: the bit pattern 0x4B0000nn with nn = code ^ 0x80
// is the float 2^23 + 128 + code, so one subtraction (exact) recovers the
// code as a float; then one IEEE product with the scale.
__device__ __forceinline__ float4 unpack_codes(uint32_t p, float scale) {
    const uint32_t b = p ^ 0x80808080u;
    constexpr float kBase = 8388736.0f;  // 2^23 + 128
    float4 o;
    o.x = (__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7440)) - kBase) * scale;
    o.y = (__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7441)) - kBase) * scale;
    o.z = (__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7442)) - kBase) * scale;
    o.w = (__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7443)) - kBase) * scale;
    return o;
}

__device__ __forceinline__ float absmax4(const float4 &v) {
    return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

__device__ __forceinline__ float4 ld_stream_f4(const float4 *p) {
    const uint4 u = ld_stream(reinterpret_cast<const uint4 *>(p));
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}

__device__ __forceinline__ void st_stream_f4(float4 *p, const float4 &v) {
    st_stream(reinterpret_cast<uint4 *>(p),
              make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w)));
}

__device__ __forceinline__ bool grouped_rows(int d, int &lpr) {
    const int nvec = d >> 2;
    if (nvec % kRowVec != 0)
        return false;
    lpr = nvec / kRowVec;
    return lpr <= 32 && (lpr & (lpr - 1)) == 0;
}

// One round of the grouped encoder: the lane's vectors v of row r (live:
// r is a row of the tile) -> the row's scale (first lane of the group) and
// the lane's codes.
__device__ __forceinline__ void encode_round(const Span &s, int d, int lpr, int l, int r, bool live,
                                             const float4 (&v)[kRowVec]) {
    float amax = 0.0f;
    if (live) {
#pragma unroll
        for (int w = 0; w < kRowVec; w++)
            amax = fmaxf(amax, absmax4(v[w]));
    }
    amax = group_max(amax, lpr);
    if (live) {
        const RowScale rs = row_scale(amax);
        if (l == 0)
            reinterpret_cast<float *>(s.scales)[r] = rs.scale;
        uint32_t q[kRowVec];
        quant_lane(v, rs, q);
        uint32_t *out = reinterpret_cast<uint32_t *>(s.dst + (int64_t)r * d) + l * kRowVec;
        if (kRowVec == 4)
            *reinterpret_cast<uint4 *>(out) = make_uint4(q[0], q[1], q[2 % kRowVec], q[3 % kRowVec]);
        else if (kRowVec == 2)
            *reinterpret_cast<uint2 *>(out) = make_uint2(q[0], q[1 % kRowVec]);
        else
#pragma unroll
            for (int w = 0; w < kRowVec; w++)
                out[w] = q[w];
    }
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

template <int kNT>
__device__ __forceinline__ void encode_grouped(const Span &s, int d, int lpr) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kWarps = kNT / 32;
    const int nvec = d >> 2;
    const int per_warp = 32 / lpr, sub = lane / lpr, l = lane % lpr;
    const int step = kWarps * per_warp;
    const float4 *src = reinterpret_cast<const float4 *>(s.src) + l * kRowVec;
    const int r0 = warp * per_warp + sub;
    // each thread stages its own vectors of the next kQ8Stages - 1 rounds in
    // shared memory with asynchronous copies (no registers held, no other
    // thread involved), waiting only on its own copy groups
    __shared__ __align__(16) float4 stage[kQ8Stages][kNT][kRowVec];
    const int rounds = (s.bytes - warp * per_warp + step - 1) / step;  // rounds this warp runs
    auto issue = [&](int k) {
        const int rr = r0 + k * step;
        if (k < rounds && rr < s.bytes) {
#pragma unroll
            for (int w = 0; w < kRowVec; w++)
                cp_async16(&stage[k % kQ8Stages][threadIdx.x][w], src + (int64_t)rr * nvec + w);
        }
        cp_async_commit();  // one group per round, empty or not
    };
#pragma unroll
    for (int k = 0; k < kQ8Stages - 1; k++)
        issue(k);
    for (int k = 0; k < rounds; k++) {
        issue(k + kQ8Stages - 1);
        cp_async_wait<kQ8Stages - 1>();  // round k's group has landed
        const int r = r0 + k * step;
        const bool live = r < s.bytes;
        float4 v[kRowVec];
        if (live) {
#pragma unroll
            for (int w = 0; w < kRowVec; w++)
                v[w] = stage[k % kQ8Stages][threadIdx.x][w];
        }
        encode_round(s, d, lpr, l, r, live, v);
    }
    cp_async_wait<0>();  // the stages are free for the next tile
}

// s.bytes rows of d values at s.src -> codes at s.dst, scales at s.scales.
template <int kNT>
__device__ __forceinline__ void encode_rows(const Span &s, int d) {
    int lpr;
    if (grouped_rows(d, lpr)) {
        encode_grouped<kNT>(s, d, lpr);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kWarps = kNT / 32;
    const int nvec = d >> 2;
    float *scales = reinterpret_cast<float *>(s.scales);
    for (int r = warp; r < s.bytes; r += kWarps) {  // other row lengths: one row per warp
        const float4 *x = reinterpret_cast<const float4 *>(s.src) + (int64_t)r * nvec;
        float amax = 0.0f;
        for (int e = lane; e < nvec; e += 32)
            amax = fmaxf(amax, absmax4(ld_stream_f4(x + e)));
        amax = group_max(amax, 32);
        const RowScale rs = row_scale(amax);
        if (lane == 0)
            scales[r] = rs.scale;
        uint32_t *q = reinterpret_cast<uint32_t *>(s.dst + (int64_t)r * d);
        for (int e = lane; e < nvec; e += 32) {
            const float4 v[1] = {ld_stream_f4(x + e)};
            uint32_t c[1];
            quant_lane(v, rs, c);
            q[e] = c[0];
        }
    }
}

// Codes at s.src (s.bytes rows of d) and scales at s.scales -> values at
// s.dst. The tile's rows are a multiple of 4 and d % 4 == 0, so its codes are
// whole 16-byte vectors, each covering one row (d a power of two >= 16) or up
// to four. kU rounds of loads are issued before their stores; with kWide the
// 64 output bytes of a vector go out as two 32-byte stores (whole sectors).
template <int kNT, bool kOneRow, int kU, bool kWide>
__device__ __forceinline__ void decode_flat(const Span &s, int d) {
    const int n = (s.bytes * d) >> 4;
    const uint4 *codes = reinterpret_cast<const uint4 *>(s.src);
    const float *scales = reinterpret_cast<const float *>(s.scales);
    float4 *x = reinterpret_cast<float4 *>(s.dst);
    const int shift = __ffs(d) - 1;
    for (int base = threadIdx.x; base < n; base += kU * kNT) {
        uint4 c[kU];
        float sc[kU][kOneRow ? 1 : 4];
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const int v = base + u * kNT;
            if (v < n) {
                c[u] = ld_stream(codes + v);
                if (kOneRow) {
                    sc[u][0] = __ldg(scales + ((v << 4) >> shift));
                } else {
#pragma unroll
                    for (int w = 0; w < 4; w++)
                        sc[u][w] = __ldg(scales + ((v << 4) + 4 * w) / d);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const int v = base + u * kNT;
            if (v < n) {
                const uint32_t w4[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
                float4 o[4];
#pragma unroll
                for (int w = 0; w < 4; w++)
                    o[w] = unpack_codes(w4[w], sc[u][kOneRow ? 0 : w]);
                if (kWide) {
#pragma unroll
                    for (int w = 0; w < 4; w += 2) {
                        u8x32 p;
                        p.lo = make_uint4(__float_as_uint(o[w].x), __float_as_uint(o[w].y), __float_as_uint(o[w].z),
                                          __float_as_uint(o[w].w));
                        p.hi = make_uint4(__float_as_uint(o[w + 1].x), __float_as_uint(o[w + 1].y),
                                          __float_as_uint(o[w + 1].z), __float_as_uint(o[w + 1].w));
                        st_stream32(reinterpret_cast<u8x32 *>(x + 4 * (int64_t)v + w), p);
                    }
                } else {
#pragma unroll
                    for (int w = 0; w < 4; w++)
                        st_stream_f4(x + 4 * (int64_t)v + w, o[w]);
                }
            }
        }
    }
}

template <int kNT>
__device__ __forceinline__ void decode_rows(const Span &s, int d) {
    if (d >= 16 && (d & (d - 1)) == 0) {
        if ((reinterpret_cast<uintptr_t>(s.dst) & 31) == 0)
            decode_flat<kNT, true, kDecUnroll, true>(s, d);
        else
            decode_flat<kNT, true, kDecUnroll, false>(s, d);
    } else {
        decode_flat<kNT, false, 1, false>(s, d);  // other row lengths: tested, not tuned
    }
}

// Vector engine: every thread of the CTA copies 32-byte (or 16-byte) vectors
// of the tile, all loads of a round issued before the matching stores.
// kU32 / kU16: vectors per thread per round on the 32- / 16-byte paths (the
// codec kernels, which run under a tighter register budget, copy with fewer).
template <bool kVec, int kCodec, int kNT = kThreads, int kU32 = LMC_VEC32_UNROLL, int kU16 = kUnroll>
__device__ __forceinline__ void copy_tiles(const Plan &P) {
    for (int64_t tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x) {
        Span s;
        const uint32_t bad = resolve<kCodec != 0>(P, tile, s);
        if (bad) {
            if (threadIdx.x == 0)
                atomicOr(P.status, bad);
            continue;
        }
        if (kCodec == 1 && s.codec == 1) {
            encode_rows<kNT>(s, P.q8_row);
        } else if (kCodec == 2 && s.codec == 2) {
            decode_rows<kNT>(s, P.q8_row);
        } else if (kVec && LMC_VEC32 &&
                   ((reinterpret_cast<uintptr_t>(s.src) | reinterpret_cast<uintptr_t>(s.dst) | (uint32_t)s.bytes) &
                    31) == 0) {
            // every load of a round is issued before its stores: up to
            // LMC_VEC32_UNROLL 32-byte vectors in flight per thread
            const u8x32 *src = reinterpret_cast<const u8x32 *>(s.src);
            u8x32 *dst = reinterpret_cast<u8x32 *>(s.dst);
            const int n = s.bytes >> 5;
            constexpr int kU = kU32;
            for (int base = threadIdx.x; base < n; base += kU * kNT) {
                u8x32 v[kU];
#pragma unroll
                for (int w = 0; w < kU; w++)
                    if (base + w * kNT < n)
                        v[w] = ld_stream32(src + base + w * kNT);
#pragma unroll
                for (int w = 0; w < kU; w++)
                    if (base + w * kNT < n)
                        st_stream32(dst + base + w * kNT, v[w]);
            }
        } else if (kVec) {
            const uint4 *src = reinterpret_cast<const uint4 *>(s.src);
            uint4 *dst = reinterpret_cast<uint4 *>(s.dst);
            const int n = s.bytes >> 4;
            for (int base = threadIdx.x; base < n; base += kU16 * kNT) {
                uint4 v[kU16];
#pragma unroll
                for (int w = 0; w < kU16; w++)
                    if (base + w * kNT < n)
                        v[w] = ld_stream(src + base + w * kNT);
#pragma unroll
                for (int w = 0; w < kU16; w++)
                    if (base + w * kNT < n)
                        st_stream(dst + base + w * kNT, v[w]);
            }
        } else {
            for (int i = threadIdx.x; i < s.bytes; i += kNT)
                s.dst[i] = s.src[i];
        }
    }
}

// Distinct names per operation (they share the body; the plan's mode says
// which side is the pool).
template <bool kVec>
__global__ void __launch_bounds__(kThreads, LMC_MIN_BLOCKS) lmc_store_kernel(const __grid_constant__ Plan P) {
    copy_tiles<kVec, 0>(P);
}
template <bool kVec>
__global__ void __launch_bounds__(kThreads, LMC_MIN_BLOCKS) lmc_load_kernel(const __grid_constant__ Plan P) {
    copy_tiles<kVec, 0>(P);
}
template <bool kVec>
__global__ void __launch_bounds__(kThreads, LMC_MIN_BLOCKS) lmc_copy_kernel(const __grid_constant__ Plan P) {
    copy_tiles<kVec, 0>(P);
}
constexpr int kEncThreads = LMC_Q8_ENC_THREADS;
constexpr int kDecThreads = LMC_Q8_DEC_THREADS;
__global__ void __launch_bounds__(kEncThreads, LMC_Q8_ENC_MIN_BLOCKS)
    lmc_store_q8_kernel(const __grid_constant__ Plan P) {
    copy_tiles<true, 1, kEncThreads, LMC_Q8_COPY_UNROLL, LMC_Q8_COPY_UNROLL>(P);
}
__global__ void __launch_bounds__(kDecThreads, LMC_Q8_DEC_MIN_BLOCKS)
    lmc_load_q8_kernel(const __grid_constant__ Plan P) {
    copy_tiles<true, 2, kDecThreads, LMC_Q8_COPY_UNROLL, LMC_Q8_COPY_UNROLL>(P);
}

// ---------------------------------------------------------------------------
// Bulk engine: one thread per CTA moves each tile global -> shared -> global
// with the bulk-copy (TMA) unit: cp.async.bulk into a shared-memory stage
// completing on an mbarrier, then cp.async.bulk back out as a bulk group.
// kStages stages form a ring, so kStages - 1 loads and the trailing stores
// are in flight per CTA. Every wait is bounded; on time-out the kernel raises
// LMC_ST_TIMEOUT, drains its own copies (bounded) and returns.
// ---------------------------------------------------------------------------
constexpr uint32_t kWaitLimit = 1u << 22;  // try_wait rounds (each may suspend)

__device__ __forceinline__ void mbar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit = kWaitLimit) {
    for (uint32_t k = 0; k < limit; k++)
        if (mbar_try_wait(bar, parity))
            return true;
    return false;
}

// Self-test of the bounded wait: one thread polls an mbarrier that nothing
// will complete (no arrival is expected, no copy targets it) and, when the
// limit runs out, reports LMC_ST_TIMEOUT like the bulk engine does.
__global__ void lmc_selftest_wait_kernel(uint32_t *status, uint32_t rounds) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0)
        return;
    mbar_init(&bar);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!mbar_wait(&bar, 0u, rounds))
        atomicOr(status, LMC_ST_TIMEOUT);
}

// Self-test of the codec's row scale: for each amax, the scale and inverse
// the encoder uses, and the IEEE quotient amax / 127 beside them.
__global__ void lmc_selftest_row_scale_kernel(const float *amax, float *scale, float *inv, float *ieee, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float a = amax[i];
        const RowScale rs = row_scale(a);
        scale[i] = rs.scale;
        inv[i] = rs.inv;
        ieee[i] = __fdiv_rn(a, 127.0f);
    }
}

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_read_all_but_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int kStages>
__device__ __forceinline__ void bulk_tiles(const Plan &P) {
    static_assert(kStages >= 2, "the ring needs a stage to fill while another drains");
    extern __shared__ __align__(128) uint8_t stage_mem[];
    __shared__ uint64_t bars[kStages];
    if (threadIdx.x != 0)
        return;
    for (int s = 0; s < kStages; s++)
        mbar_init(&bars[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

    Span span[kStages];
    int32_t state[kStages];  // -1: no tile left, 0: skipped tile, 1: load in flight, 2: stored
    uint32_t parity = 0;     // bit s: phase parity to wait for on stage s
    int64_t next = blockIdx.x;

    auto issue = [&](int s) {
        if (next >= P.total_tiles) {
            state[s] = -1;
            return;
        }
        const uint32_t bad = resolve<false>(P, next, span[s]);
        next += gridDim.x;
        if (bad) {
            atomicOr(P.status, bad);
            state[s] = 0;
            return;
        }
        uint8_t *buf = stage_mem + (size_t)s * kTileBytes;
        mbar_arrive_expect(&bars[s], (uint32_t)span[s].bytes);
        bulk_load(buf, span[s].src, (uint32_t)span[s].bytes, &bars[s]);
        state[s] = 1;
    };

    for (int s = 0; s < kStages - 1; s++)
        issue(s);
    state[kStages - 1] = -1;
    bool timed_out = false;
    for (int64_t i = 0;; i++) {
        const int s = (int)(i % kStages);  // stage holding this CTA's i-th tile
        if (state[s] < 0)
            break;
        if (state[s] == 1) {
            if (!mbar_wait(&bars[s], (parity >> s) & 1u)) {
                timed_out = true;
                break;
            }
            parity ^= 1u << s;
            bulk_store(span[s].dst, stage_mem + (size_t)s * kTileBytes, (uint32_t)span[s].bytes);
            state[s] = 2;
        }
        bulk_commit();
        // all stores but the one just issued have read their stage: the
        // stage of tile i - 1 is free for tile i + kStages - 1
        bulk_wait_read_all_but_one();
        issue((int)((i + kStages - 1) % kStages));
    }
    if (timed_out) {
        atomicOr(P.status, LMC_ST_TIMEOUT);
        // let the loads still in flight land before the CTA's shared memory goes away
        for (int s = 0; s < kStages; s++)
            if (state[s] == 1)
                mbar_wait(&bars[s], (parity >> s) & 1u);
    }
    bulk_wait_all();
}

template <int kStages>
__global__ void __launch_bounds__(32) lmc_store_bulk_kernel(const __grid_constant__ Plan P) {
    bulk_tiles<kStages>(P);
}
template <int kStages>
__global__ void __launch_bounds__(32) lmc_load_bulk_kernel(const __grid_constant__ Plan P) {
    bulk_tiles<kStages>(P);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

int sm_count() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return -1;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev)
        cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return -1;
        cache[dev] = n;
    }
    return cache[dev];
}

bool aligned16(int64_t x) { return (x & 15) == 0; }

// Appends a layer entry: `pages` pages of `d` per object. The pages lie back
// to back from the object's current offset `obj`, which advances past them;
// with rec_stride > 0 page j lies at obj + j * rec_stride instead (the page
// part of interleaved records) and the caller advances obj.
int add_entry(Plan &P, int &ne, const lmc_layer_desc &d, int64_t pages, bool last, int64_t &obj,
              int64_t &tiles, bool &vec, int64_t rec_stride = 0) {
    if (ne >= kMaxEntries)
        return LMC_ERR_INVALID_ARG;
    if (d.real_bytes > INT32_MAX - kTileBytes)
        return LMC_ERR_INVALID_ARG;  // one page must stay below 2 GiB
    const int32_t seg = (int32_t)d.real_bytes;
    const int32_t pieces = (seg + kTileBytes - 1) / kTileBytes;
    int32_t tb = (seg + pieces - 1) / pieces;
    const int32_t align = seg % 32 == 0 ? 32 : 16;  // keep 32-byte pages in 32-byte pieces
    tb = (tb + align - 1) / align * align;          // the last piece is shorter
    Entry &E = P.entries[ne++];
    E.pool_base = d.base;
    E.pool_stride = d.stride;
    E.obj_off = obj;
    E.seg_bytes = seg;
    E.tile_bytes = tb;
    E.tiles_per_seg = (seg + tb - 1) / tb;
    E.tile_start = (int32_t)tiles;
    E.kda = d.kind == LMC_LAYER_KDA;
    E.codec = 0;
    E.last = last;
    E.kv = (uint8_t)d.kv_group;
    E.obj_stride = rec_stride > 0 ? (int32_t)rec_stride : seg;
    int64_t add;
    if (rec_stride > INT32_MAX || (rec_stride == 0 && (!lmc::mul_ok(pages, seg, &add) || !lmc::add_ok(obj, add, &obj))))
        return LMC_ERR_OVERFLOW;
    tiles += pages * E.tiles_per_seg;
    if (tiles > INT32_MAX)
        return LMC_ERR_OVERFLOW;
    vec = vec && aligned16(d.base) && aligned16(d.stride) && aligned16(seg);
    return LMC_OK;
}

// Appends the codec entry of a KDA layer: for each of `pages` snapshots per
// object, the recurrent state after the conv bytes, encoded as the scales
// then the codes of an INT8 record at obj_off + j * rec_stride.
int add_codec_entry(Plan &P, int &ne, const lmc_layer_desc &d, const lmc_layer_spec &spec, int64_t pages,
                    bool last, int64_t obj_off, int64_t rec_stride, int64_t &tiles, bool &vec) {
    if (ne >= kMaxEntries)
        return LMC_ERR_INVALID_ARG;
    const int64_t row = P.q8_row;
    const int64_t rows = spec.rec_bytes / (4 * row);
    if (rows > INT32_MAX || spec.conv_bytes > INT32_MAX || rec_stride > INT32_MAX)
        return LMC_ERR_INVALID_ARG;
    // rows per tile: a multiple of 4, so every tile's codes and scales start
    // on a 16-byte boundary
    const int32_t per_tile = (int32_t)std::max<int64_t>(4, kQ8TileBytes / (4 * row) / 4 * 4);
    Entry &E = P.entries[ne++];
    E.pool_base = d.base + spec.conv_bytes;  // the state starts after the conv bytes
    E.pool_stride = d.stride;
    E.obj_off = obj_off;
    E.obj_stride = (int32_t)rec_stride;
    E.seg_bytes = (int32_t)rows;  // a codec entry counts rows
    E.tile_bytes = per_tile;
    E.tiles_per_seg = (int32_t)((rows + per_tile - 1) / per_tile);
    E.tile_start = (int32_t)tiles;
    E.kda = 1;
    E.codec = 1;
    E.last = last;
    E.kv = (uint8_t)d.kv_group;
    tiles += pages * E.tiles_per_seg;
    // the rows are read and written as 16-byte vectors
    vec = vec && aligned16(d.base) && aligned16(d.stride) && aligned16(spec.conv_bytes);
    return tiles > INT32_MAX ? LMC_ERR_OVERFLOW : LMC_OK;
}

// Adds a group of `n` items to the plan's tile space.
int close_group(Plan &P, int ne, int first_entry, const void *items, int64_t n, int64_t obj, int64_t tiles,
                int64_t &total) {
    if (P.num_groups >= kMaxGroups)
        return LMC_ERR_INVALID_ARG;
    Group &G = P.groups[P.num_groups++];
    G.items = items;
    G.num_items = n;
    G.first_entry = first_entry;
    G.num_entries = ne - first_entry;
    G.obj_bytes = obj;
    G.tiles_per_obj = (int32_t)tiles;
    G.tile_begin = total;
    int64_t add;
    if (!lmc::mul_ok(n, tiles, &add) || !lmc::add_ok(total, add, &total))
        return LMC_ERR_OVERFLOW;
    return LMC_OK;
}

// Object geometry of one call: an object covers `nb` block positions from
// job.chunk * pos_mul; KDA layers give the last block's snapshot, or one per
// block with kda_every.
struct Shape {
    int64_t nb;
    int32_t pos_mul;
    bool kda_every;
    int32_t q8_row;  // > 0: KDA snapshots as INT8 records with rows of q8_row values
};

// Host-side validation and launch plan of a store or load.
int build_object_plan(const lmc_layout *L, const Shape &sh, const void *pool, const lmc_batch *b,
                      const void *arena, int64_t arena_bytes, uint32_t *status, Mode mode, Plan &P,
                      bool &vec) {
    if (b == nullptr || status == nullptr)
        return LMC_ERR_INVALID_ARG;
    if (((uintptr_t)status & 3) != 0)
        return LMC_ERR_ALIGN;
    const int nkv = (int)L->kv_group_kind.size();
    const int nog = (int)L->object_group_layers.size();
    if (b->num_requests < 0 || b->num_kv_groups != nkv || b->num_object_groups != nog ||
        arena_bytes < 0 || (nkv > 0 && b->tables == nullptr) || b->num_jobs == nullptr ||
        b->jobs == nullptr)
        return LMC_ERR_INVALID_ARG;
    if (nkv > kMaxKv || nog > kMaxGroups)
        return LMC_ERR_INVALID_ARG;

    std::memset(&P, 0, sizeof(P));
    P.pos_mul = sh.pos_mul;
    P.last_pos = (int32_t)(sh.nb - 1);
    P.q8_row = sh.q8_row;
    P.num_requests = b->num_requests;
    P.num_blocks = L->num_blocks;
    P.arena_bytes = arena_bytes;
    P.status = status;
    P.mode = mode;
    for (int k = 0; k < nkv; k++) {
        const lmc_block_table &t = b->tables[k];
        if (t.num_cols < 0 || t.row_stride < t.num_cols ||
            (b->num_requests > 0 && t.num_cols > 0 && t.table == nullptr))
            return LMC_ERR_INVALID_ARG;
        P.tables[k] = Table{t.table, t.row_stride, t.num_cols};
    }

    vec = aligned16((int64_t)(uintptr_t)pool) && aligned16((int64_t)(uintptr_t)arena);
    int64_t total = 0;
    int ne = 0;
    for (int og = 0; og < nog; og++) {
        const int64_t nj = b->num_jobs[og];
        if (nj < 0 || (nj > 0 && b->jobs[og] == nullptr))
            return LMC_ERR_INVALID_ARG;
        if (nj == 0)
            continue;
        const int first = ne;
        int64_t obj = 0, tiles = 0;
        for (int32_t i : L->object_group_layers[og]) {
            const lmc_layer_desc &d = L->desc[i];
            const bool last_only = d.kind == LMC_LAYER_KDA && !sh.kda_every;
            int rc;
            if (d.kind == LMC_LAYER_KDA && sh.q8_row > 0) {
                // one INT8 record per stored snapshot, back to back: the conv
                // window as is, then the state's scales and codes
                const lmc_layer_spec &spec = L->specs[i];
                const int64_t pages = last_only ? 1 : sh.nb;
                const int64_t rows = spec.rec_bytes / (4 * (int64_t)sh.q8_row);
                const int64_t record = spec.conv_bytes + 4 * rows + rows * (int64_t)sh.q8_row;
                lmc_layer_desc conv = d;
                conv.real_bytes = spec.conv_bytes;
                int64_t at = obj, add = 0;
                rc = conv.real_bytes > 0 ? add_entry(P, ne, conv, pages, last_only, at, tiles, vec, record) : LMC_OK;
                if (rc == LMC_OK)
                    rc = add_codec_entry(P, ne, d, spec, pages, last_only, obj + spec.conv_bytes, record, tiles, vec);
                if (rc == LMC_OK && (!lmc::mul_ok(pages, record, &add) || !lmc::add_ok(obj, add, &obj)))
                    rc = LMC_ERR_OVERFLOW;
            } else {
                rc = add_entry(P, ne, d, last_only ? 1 : sh.nb, last_only, obj, tiles, vec);
            }
            if (rc != LMC_OK)
                return rc;
        }
        const int rc = close_group(P, ne, first, b->jobs[og], nj, obj, tiles, total);
        if (rc != LMC_OK)
            return rc;
    }
    P.total_tiles = total;
    if (total > 0 && (pool == nullptr || arena == nullptr))
        return LMC_ERR_INVALID_ARG;
    P.src_base = static_cast<const uint8_t *>(mode == kStore ? pool : arena);
    P.dst_base = static_cast<uint8_t *>(const_cast<void *>(mode == kStore ? arena : pool));
    return LMC_OK;
}

int launch_plan(const Plan &P, bool vec, void *stream) {
    if (P.total_tiles == 0)
        return LMC_OK;
    const int sms = sm_count();
    if (sms <= 0)
        return LMC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (vec && kEngine == 1 && P.mode != kCopy && P.q8_row == 0) {
        // persistent: kBulkCtasPerSm CTAs per SM, each a ring of stages
        const size_t smem = (size_t)kBulkStages * kTileBytes;
        auto kern = P.mode == kStore ? lmc_store_bulk_kernel<kBulkStages> : lmc_load_bulk_kernel<kBulkStages>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LMC_ERR_CUDA;
        const unsigned grid = (unsigned)std::min<int64_t>(P.total_tiles, (int64_t)sms * kBulkCtasPerSm);
        kern<<<grid, 32, smem, s>>>(P);
    } else {
        // one CTA per tile, capped; the kernel strides over the rest
        const unsigned grid = (unsigned)std::min<int64_t>(P.total_tiles, (int64_t)sms * 2048);
        if (P.q8_row > 0) {
            if (P.mode == kStore)
                lmc_store_q8_kernel<<<grid, kEncThreads, 0, s>>>(P);
            else
                lmc_load_q8_kernel<<<grid, kDecThreads, 0, s>>>(P);
            return cudaGetLastError() == cudaSuccess ? LMC_OK : LMC_ERR_CUDA;
        }
        void (*kern)(const Plan);
        if (P.mode == kStore)
            kern = vec ? lmc_store_kernel<true> : lmc_store_kernel<false>;
        else if (P.mode == kLoad)
            kern = vec ? lmc_load_kernel<true> : lmc_load_kernel<false>;
        else
            kern = vec ? lmc_copy_kernel<true> : lmc_copy_kernel<false>;
        kern<<<grid, kThreads, 0, s>>>(P);
    }
    return cudaGetLastError() == cudaSuccess ? LMC_OK : LMC_ERR_CUDA;
}

int chunk_shape(const lmc_layout *L, int64_t chunk, Shape &sh) {
    if (L == nullptr)
        return LMC_ERR_INVALID_ARG;
    if (chunk <= 0 || chunk % L->block_size != 0)
        return LMC_ERR_NOT_MULTIPLE;
    const int64_t m = chunk / L->block_size;
    if (m > INT32_MAX)
        return LMC_ERR_OVERFLOW;
    sh = Shape{m, (int32_t)m, false, 0};
    return LMC_OK;
}

int block_shape(const lmc_layout *L, int64_t nb, int32_t kda_mode, Shape &sh) {
    if (L == nullptr || nb <= 0 || nb > INT32_MAX ||
        (kda_mode != LMC_KDA_LAST_BLOCK && kda_mode != LMC_KDA_EVERY_BLOCK))
        return LMC_ERR_INVALID_ARG;
    sh = Shape{nb, 1, kda_mode == LMC_KDA_EVERY_BLOCK, 0};
    return LMC_OK;
}

int run_objects(const lmc_layout *L, const Shape &sh, const void *pool, const lmc_batch *b, const void *arena,
                int64_t arena_bytes, uint32_t *status, void *stream, Mode mode) {
    Plan P;
    bool vec = false;
    const int rc = build_object_plan(L, sh, pool, b, arena, arena_bytes, status, mode, P, vec);
    if (rc != LMC_OK)
        return rc;
    if (sh.q8_row > 0 && !vec)
        return LMC_ERR_ALIGN;  // the codec reads and writes rows as 16-byte vectors
    return launch_plan(P, vec, stream);
}

// Row lengths the codec accepts: 4 <= d <= 512, d % 4 == 0, every KDA
// layer's recurrent state a whole number of rows and a multiple of 4 rows,
// and its conv bytes a multiple of 16: every record stays a multiple of 16
// bytes, so the rows behind it remain 16-byte aligned.
int q8_check(const lmc_layout *L, int64_t d) {
    if (d < 4 || d > 512 || d % 4 != 0)
        return LMC_ERR_INVALID_ARG;
    for (const lmc_layer_spec &spec : L->specs)
        if (spec.kind == LMC_LAYER_KDA && (spec.rec_bytes % (4 * d) != 0 || (spec.rec_bytes / (4 * d)) % 4 != 0 ||
                                           spec.conv_bytes % 16 != 0))
            return LMC_ERR_INVALID_ARG;
    return LMC_OK;
}

int q8_shape(const lmc_layout *L, int64_t chunk, int64_t d, Shape &sh) {
    int rc = chunk_shape(L, chunk, sh);
    if (rc == LMC_OK)
        rc = q8_check(L, d);
    sh.q8_row = rc == LMC_OK ? (int32_t)d : 0;
    return rc;
}

int q8_block_shape(const lmc_layout *L, int64_t nb, int32_t kda_mode, int64_t d, Shape &sh) {
    int rc = block_shape(L, nb, kda_mode, sh);
    if (rc == LMC_OK)
        rc = q8_check(L, d);
    sh.q8_row = rc == LMC_OK ? (int32_t)d : 0;
    return rc;
}

// Bytes of one object of `og` with INT8 KDA records: a paged layer's nb
// pages, a KDA layer's one (or, every block, nb) records.
int object_bytes_q8(const lmc_layout *L, const Shape &sh, int32_t og, int64_t *out) {
    if (out == nullptr || og < 0 || (size_t)og >= L->object_group_layers.size())
        return LMC_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int32_t i : L->object_group_layers[og]) {
        const lmc_layer_spec &spec = L->specs[i];
        int64_t part;
        if (spec.kind == LMC_LAYER_KDA) {
            const int64_t rows = spec.rec_bytes / (4 * (int64_t)sh.q8_row);
            const int64_t record = spec.conv_bytes + 4 * rows + rows * (int64_t)sh.q8_row;
            if (!lmc::mul_ok(sh.kda_every ? sh.nb : 1, record, &part))
                return LMC_ERR_OVERFLOW;
        } else if (!lmc::mul_ok(sh.nb, L->desc[i].real_bytes, &part)) {
            return LMC_ERR_OVERFLOW;
        }
        if (!lmc::add_ok(total, part, &total))
            return LMC_ERR_OVERFLOW;
    }
    *out = total;
    return LMC_OK;
}

}  // namespace

extern "C" int lmc_store(const lmc_layout *layout, int64_t chunk_size, const void *pool,
                         const lmc_batch *batch, void *arena, int64_t arena_bytes, uint32_t *status,
                         void *stream) {
    Shape sh;
    const int rc = chunk_shape(layout, chunk_size, sh);
    return rc != LMC_OK ? rc : run_objects(layout, sh, pool, batch, arena, arena_bytes, status, stream, kStore);
}

extern "C" int lmc_load(const lmc_layout *layout, int64_t chunk_size, void *pool,
                        const lmc_batch *batch, const void *arena, int64_t arena_bytes,
                        uint32_t *status, void *stream) {
    Shape sh;
    const int rc = chunk_shape(layout, chunk_size, sh);
    return rc != LMC_OK ? rc : run_objects(layout, sh, pool, batch, arena, arena_bytes, status, stream, kLoad);
}

extern "C" int lmc_store_blocks(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                                const void *pool, const lmc_batch *batch, void *arena, int64_t arena_bytes,
                                uint32_t *status, void *stream) {
    Shape sh;
    const int rc = block_shape(layout, blocks_per_object, kda_mode, sh);
    return rc != LMC_OK ? rc : run_objects(layout, sh, pool, batch, arena, arena_bytes, status, stream, kStore);
}

extern "C" int lmc_load_blocks(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                               void *pool, const lmc_batch *batch, const void *arena, int64_t arena_bytes,
                               uint32_t *status, void *stream) {
    Shape sh;
    const int rc = block_shape(layout, blocks_per_object, kda_mode, sh);
    return rc != LMC_OK ? rc : run_objects(layout, sh, pool, batch, arena, arena_bytes, status, stream, kLoad);
}

extern "C" int lmc_copy_blocks(const lmc_layout *L, void *pool, const lmc_copy_batch *b, uint32_t *status,
                               void *stream) {
    if (L == nullptr || b == nullptr || status == nullptr)
        return LMC_ERR_INVALID_ARG;
    if (((uintptr_t)status & 3) != 0)
        return LMC_ERR_ALIGN;
    const int nkv = (int)L->kv_group_kind.size();
    if (b->num_kv_groups != nkv || nkv > kMaxGroups || b->pairs == nullptr || b->num_pairs == nullptr)
        return LMC_ERR_INVALID_ARG;
    for (int g = 0; g < nkv; g++)
        if (b->num_pairs[g] < 0 || (b->num_pairs[g] > 0 && b->pairs[g] == nullptr))
            return LMC_ERR_INVALID_ARG;
    // the pairs run concurrently: refuse a batch whose copies would race
    if (const int rc = lmc::check_copy_pairs(L, b); rc != LMC_OK)
        return rc;
    Plan P;
    std::memset(&P, 0, sizeof(P));
    P.num_blocks = L->num_blocks;
    P.status = status;
    P.mode = kCopy;
    bool vec = aligned16((int64_t)(uintptr_t)pool);
    int64_t total = 0;
    int ne = 0;
    for (int g = 0; g < nkv; g++) {
        const int64_t n = b->num_pairs[g];
        if (n < 0 || (n > 0 && b->pairs[g] == nullptr))
            return LMC_ERR_INVALID_ARG;
        if (n == 0)
            continue;
        const int first = ne;
        int64_t obj = 0, tiles = 0;
        for (size_t i = 0; i < L->desc.size(); i++) {
            if (L->desc[i].kv_group != g)
                continue;
            const int rc = add_entry(P, ne, L->desc[i], 1, false, obj, tiles, vec);
            if (rc != LMC_OK)
                return rc;
        }
        const int rc = close_group(P, ne, first, b->pairs[g], n, obj, tiles, total);
        if (rc != LMC_OK)
            return rc;
    }
    P.total_tiles = total;
    if (total > 0 && pool == nullptr)
        return LMC_ERR_INVALID_ARG;
    P.src_base = static_cast<const uint8_t *>(pool);
    P.dst_base = static_cast<uint8_t *>(pool);
    return launch_plan(P, vec, stream);
}

extern "C" int lmc_store_q8(const lmc_layout *layout, int64_t chunk_size, int64_t row_elems, const void *pool,
                            const lmc_batch *batch, void *arena, int64_t arena_bytes, uint32_t *status,
                            void *stream) {
    Shape sh;
    const int rc = q8_shape(layout, chunk_size, row_elems, sh);
    return rc != LMC_OK ? rc : run_objects(layout, sh, pool, batch, arena, arena_bytes, status, stream, kStore);
}

extern "C" int lmc_load_q8(const lmc_layout *layout, int64_t chunk_size, int64_t row_elems, void *pool,
                           const lmc_batch *batch, const void *arena, int64_t arena_bytes, uint32_t *status,
                           void *stream) {
    Shape sh;
    const int rc = q8_shape(layout, chunk_size, row_elems, sh);
    return rc != LMC_OK ? rc : run_objects(layout, sh, pool, batch, arena, arena_bytes, status, stream, kLoad);
}

extern "C" int lmc_object_bytes_q8(const lmc_layout *layout, int64_t chunk_size, int64_t row_elems,
                                   int32_t object_group, int64_t *out) {
    Shape sh;
    const int rc = q8_shape(layout, chunk_size, row_elems, sh);
    return rc != LMC_OK ? rc : object_bytes_q8(layout, sh, object_group, out);
}

extern "C" int lmc_store_blocks_q8(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                                   int64_t row_elems, const void *pool, const lmc_batch *batch, void *arena,
                                   int64_t arena_bytes, uint32_t *status, void *stream) {
    Shape sh;
    const int rc = q8_block_shape(layout, blocks_per_object, kda_mode, row_elems, sh);
    return rc != LMC_OK ? rc : run_objects(layout, sh, pool, batch, arena, arena_bytes, status, stream, kStore);
}

extern "C" int lmc_load_blocks_q8(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                                  int64_t row_elems, void *pool, const lmc_batch *batch, const void *arena,
                                  int64_t arena_bytes, uint32_t *status, void *stream) {
    Shape sh;
    const int rc = q8_block_shape(layout, blocks_per_object, kda_mode, row_elems, sh);
    return rc != LMC_OK ? rc : run_objects(layout, sh, pool, batch, arena, arena_bytes, status, stream, kLoad);
}

extern "C" int lmc_object_bytes_blocks_q8(const lmc_layout *layout, int64_t blocks_per_object, int32_t kda_mode,
                                          int64_t row_elems, int32_t object_group, int64_t *out) {
    Shape sh;
    const int rc = q8_block_shape(layout, blocks_per_object, kda_mode, row_elems, sh);
    return rc != LMC_OK ? rc : object_bytes_q8(layout, sh, object_group, out);
}

extern "C" int lmc_selftest_row_scale(const float *amax, float *scale, float *inv, float *ieee, int64_t n,
                                      void *stream) {
    if (n < 0 || (n > 0 && (amax == nullptr || scale == nullptr || inv == nullptr || ieee == nullptr)))
        return LMC_ERR_INVALID_ARG;
    if ((((uintptr_t)amax | (uintptr_t)scale | (uintptr_t)inv | (uintptr_t)ieee) & 3) != 0)
        return LMC_ERR_ALIGN;
    if (n == 0)
        return LMC_OK;
    const int sms = sm_count();
    if (sms <= 0)
        return LMC_ERR_CUDA;
    const unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, (int64_t)sms * 8);
    lmc_selftest_row_scale_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(amax, scale, inv, ieee, n);
    return cudaGetLastError() == cudaSuccess ? LMC_OK : LMC_ERR_CUDA;
}

extern "C" int lmc_selftest_wait(uint32_t *status, int64_t rounds, void *stream) {
    if (status == nullptr || rounds <= 0 || rounds > (int64_t)kWaitLimit)
        return LMC_ERR_INVALID_ARG;
    if (((uintptr_t)status & 3) != 0)
        return LMC_ERR_ALIGN;
    lmc_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, (uint32_t)rounds);
    return cudaGetLastError() == cudaSuccess ? LMC_OK : LMC_ERR_CUDA;
}

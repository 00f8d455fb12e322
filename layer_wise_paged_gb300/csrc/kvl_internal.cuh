// kvl_internal.cuh -- internals shared by the plan and copy translation units of
// libkvl.so: the plan's device layout, status recording, and host-side checks.
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "kvl.h"

namespace kvl {

constexpr uint32_t kPlanMagic = 0x4b564c32u;  // "KVL2"
constexpr int kOps = 4;  // slice, merge-scatter, gather, scatter-back
constexpr int kMaxDevices = 64;

// Start of a plan (the header section is padded to 256 bytes).
struct PlanHeader {
    int32_t status;              // 0: KVL_* code, the largest recorded wins
    uint32_t magic;              // 4: kPlanMagic once built
    int32_t n_req;               // 8
    int32_t check_injective;     // 12
    int64_t n_items;             // 16: sum over requests of ceil(T_all / B)
    int64_t n_tokens;            // 24: sum of T_all
    int64_t n_hit;               // 32: sum of T_hit
    int32_t scan_status;         // 40: status after the request scan (the fill reads it)
    int32_t n_layers;            // 44: L the plan was built for (sizes the counters)
    int64_t pool_blocks;         // 48: N the plan was built for
    int64_t block_tokens;        // 56: B the plan was built for
    unsigned long long detail[8];  // 64: per status code, smallest detail recorded
    const void *reqs;            // 128: the request array the plan was built from
    const void *tables;          // 136: the block tables the plan was built from
    int32_t map_chunk;           // 144: bytes per chunk of a tensor-map row (0: no maps)
    int32_t n_planes;            // 148: P the plan was built for
    int32_t plane_row_bytes;     // 152: Rp the plan was built for
    int32_t pad0;                // 156
};
static_assert(sizeof(PlanHeader) == 160, "plan header layout");
static_assert(sizeof(kvl_request) == 112, "kvl_request layout");

__host__ __device__ inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// One work item resolved once by the plan (128 bytes, 32 words: a warp loads it with
// one coalesced request, a word per lane).  Addresses are those of layer 0; a layer
// adds l times the matching layer stride.
struct ItemRec {
    uint64_t hit_base;    //  0: hit_src + sb(j)*hit_block_stride (0: no hit rows)
    int64_t hit_ts;       //  2: hit token stride
    int64_t hit_ls;       //  4: hit layer stride
    uint64_t miss_base;   //  6: miss row of slot 0: miss_src + (j*B - T_hit)*miss_ts
    int64_t miss_ts;      //  8
    int64_t miss_ls;      // 10
    uint64_t obj_base;    // 12: objects + j*obj_block_stride (0: no objects)
    int64_t obj_ps;       // 14: object plane stride
    int64_t obj_ls;       // 16: object layer stride
    int64_t hit_row;      // 18: row of hit_out holding slot 0 (hit_off[r] + j*B)
    int64_t tok_row;      // 20: row of complete_out holding slot 0 (tok_off[r] + j*B)
    int32_t pool_block;   // 22: table entry
    int32_t n_hit;        // 23: slots that are hit tokens
    int32_t n_valid;      // 24: slots that are tokens (T_all - j*B, at most B)
    int32_t req;          // 25
    int32_t hit_blk_crd;  // 26: block coordinate of the hit rows in the request's hit map
    int32_t hit_tok_crd;  // 27: token coordinate of slot 0 in the hit map
    int32_t miss_tok_crd; // 28: token coordinate of slot 0 in the miss map (j*B - T_hit)
    int32_t map_flags;    // 29: kMap* bits: which of the request's tensor maps exist
    int32_t pad[2];       // 30
};
static_assert(sizeof(ItemRec) == 128, "item record layout");

// Work-claim counter of one (layer, op): the next claim's number (0 between launches).
struct ClaimCounter {
    uint32_t next;
    uint32_t reserved;  // kept 0: holds the counter section at 8 bytes per (layer, op)
};

constexpr size_t kRecordsOffset = 256;  // the item records start right after the header

// Shared-memory stage of the copy kernels: one segment of rows, at most this long.
constexpr int kStageBytes = 32 * 1024;

// Tensor maps.  A request's strided row sources (its hit rows, read a plane at a time
// by the merge-scatter or a whole row at a time by the slice, and its miss rows) are
// also described by tensor maps that the plan builds on the device, so that a
// segment of rows from one source is one tiled bulk-tensor load instead of one bulk
// load per row.  Each map is a 5-D view of the source with 8-byte elements:
//   dim 0  bytes of one chunk of a token row (map_chunk / 8 elements)
//   dim 1  chunks of the token row (R / map_chunk of them; plane p starts at chunk
//          p * Rp / map_chunk)
//   dim 2, dim 3  tokens and layers, the one with the smaller stride first
//   dim 4  full blocks of a block-table source (extent 1 otherwise)
// The box is one plane row (merge, miss) or one token row (slice) wide and as many
// token rows high as a segment holds, so its bytes land in the stage as the per-row
// loads would place them.  Each source has a map of each of two box heights: a whole
// segment, and the rows a block has left after its whole segments (its tail: B mod
// the segment rows, when that is not 0).  Extents are exactly the rows the request
// declares, so no coordinate reaches memory the per-row loads could not.
constexpr int kMapBytes = 128;
enum MapKind {
    MAP_HIT = 0,         // hit plane rows (merge-scatter), whole segments
    MAP_SLICE = 1,       // hit token rows (slice), whole segments
    MAP_MISS = 2,        // miss plane rows (merge-scatter), whole segments
    MAP_HIT_TAIL = 3,    // the same three sources, block tails
    MAP_SLICE_TAIL = 4,
    MAP_MISS_TAIL = 5,
};
constexpr int kMapsPerReq = 6;
constexpr int kMapTail = MAP_HIT_TAIL - MAP_HIT;  // a kind's tail kind is kind + kMapTail
// Record flags: bit `kind` says the request's map of that kind exists; the hit maps
// (and the miss maps) share one view of their source, so one dim order each.
__host__ __device__ constexpr int32_t map_bit(int kind) { return int32_t(1) << kind; }
constexpr int32_t kMapHitLayerFirst = 64;   // hit maps order dims 2, 3 as (layer, token)
constexpr int32_t kMapMissLayerFirst = 128; // miss maps order dims 2, 3 as (layer, token)

// Bytes per chunk of a tensor-map row for plane rows of Rp bytes: the largest
// multiple of 16 that divides Rp and is at most 2 KiB (a box row holds at most 256
// elements of 8 bytes).
__host__ __device__ inline int32_t map_chunk_bytes(int32_t Rp)
{
    for (int32_t c = (Rp < 2048 ? Rp : 2048) & ~15; c >= 16; c -= 16)
        if (Rp % c == 0) return c;
    return 0;
}

// Token rows per segment of an op whose rows are `row_bytes` wide: a whole block,
// or as many rows as a stage holds.
__host__ __device__ inline int32_t segment_rows(int32_t B, int32_t row_bytes)
{
    const int32_t m = kStageBytes / row_bytes;
    return B < m ? B : m;
}

// Rows of a whole block left after its whole segments (0: segments divide blocks).
__host__ __device__ inline int32_t segment_tail_rows(int32_t B, int32_t row_bytes)
{
    const int32_t m = segment_rows(B, row_bytes);
    return m > 0 ? B % m : 0;
}

// Byte offsets of the plan's sections (see kvl_plan_layout).
struct PlanLayout {
    size_t off[11];
    __host__ __device__ PlanLayout() {}
};

__host__ __device__ inline PlanLayout plan_layout(int32_t n_req, int64_t pool_blocks, int32_t n_layers)
{
    PlanLayout p;
    size_t n1 = size_t(n_req < 0 ? 0 : n_req) + 1;
    size_t cap = size_t(pool_blocks < 0 ? 0 : pool_blocks);
    size_t L = size_t(n_layers < 0 ? 0 : n_layers);
    // Placement: the item records come first, at a fixed offset, so a copy kernel can
    // address its first record before it has read the header; the sections that
    // depend on n_req follow; the bitmap is last.
    p.off[0] = 0;
    p.off[6] = kRecordsOffset;                                        // item records
    p.off[4] = p.off[6] + round256(cap * sizeof(ItemRec));           // item_req
    p.off[5] = p.off[4] + round256(cap * 4);                         // item_blk
    p.off[7] = p.off[5] + round256(cap * 4);                         // claim counters
    p.off[1] = p.off[7] + round256(L * kOps * sizeof(ClaimCounter)); // tok_off
    p.off[2] = p.off[1] + round256(n1 * 8);                          // hit_off
    p.off[3] = p.off[2] + round256(n1 * 8);                          // blk_off
    // tensor maps: kMapsPerReq per request, plus slack to start them on a 128-byte
    // boundary (the plan itself need only be 16-byte aligned), then each request's
    // map flags (int32)
    p.off[10] = p.off[3] + round256(n1 * 8);                         // tensor maps
    p.off[8] = p.off[10] + round256((n1 - 1) * (kMapsPerReq * kMapBytes + 4) + kMapBytes);  // bitmap
    p.off[9] = p.off[8] + round256(((cap + 31) / 32) * 4);           // end
    return p;
}

// Device view of a built plan.
struct PlanView {
    PlanHeader *hdr;
    int64_t *tok_off;
    int64_t *hit_off;
    int64_t *blk_off;
    int32_t *item_req;
    int32_t *item_blk;
    ItemRec *items;
    ClaimCounter *counters;  // [L][kOps]
    uint32_t *bitmap;
    uint8_t *maps;           // [n_req][kMapsPerReq] tensor maps, 128-byte aligned
    int32_t *map_flags;      // [n_req] kMap* flags of each request, after the maps
};

__host__ __device__ inline PlanView plan_view(void *d_plan, int32_t n_req, int64_t pool_blocks,
                                              int32_t n_layers)
{
    PlanLayout l = plan_layout(n_req, pool_blocks, n_layers);
    char *b = static_cast<char *>(d_plan);
    PlanView v;
    v.hdr = reinterpret_cast<PlanHeader *>(b);
    v.tok_off = reinterpret_cast<int64_t *>(b + l.off[1]);
    v.hit_off = reinterpret_cast<int64_t *>(b + l.off[2]);
    v.blk_off = reinterpret_cast<int64_t *>(b + l.off[3]);
    v.item_req = reinterpret_cast<int32_t *>(b + l.off[4]);
    v.item_blk = reinterpret_cast<int32_t *>(b + l.off[5]);
    v.items = reinterpret_cast<ItemRec *>(b + l.off[6]);
    v.counters = reinterpret_cast<ClaimCounter *>(b + l.off[7]);
    v.bitmap = reinterpret_cast<uint32_t *>(b + l.off[8]);
    v.maps = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(b + l.off[10]) + 127) &
                                         ~uintptr_t(127));
    v.map_flags = reinterpret_cast<int32_t *>(v.maps + size_t(n_req < 0 ? 0 : n_req) * kMapsPerReq * kMapBytes);
    return v;
}

// Record a device-side error: the largest code wins, and each code keeps the
// smallest detail it was given.
__device__ __forceinline__ void record_error(PlanHeader *h, int code, unsigned long long detail)
{
    atomicMax(&h->status, code);
    atomicMin(&h->detail[code], detail);
}

__host__ __device__ __forceinline__ bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b)
{
    return (a + b - 1) / b;
}

// Host-side geometry check shared by every entry point.
inline kvl_status check_geom(const kvl_geom *g)
{
    if (!g) return KVL_EINVAL;
    if (g->n_layers <= 0 || g->n_planes <= 0 || g->block_tokens <= 0 ||
        g->plane_row_bytes <= 0 || g->pool_blocks <= 0)
        return KVL_EINVAL;
    if (g->pool_blocks > INT32_MAX) return KVL_EINVAL;  // block ids are int32
    if (g->plane_row_bytes % 16) return KVL_EALIGN;
    return KVL_OK;
}

// SM count of the current device (cached per device).
// SMs of the current device, cached per device (host threads may call concurrently:
// each may query the attribute once and store the same value).
inline int sm_count()
{
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// The current CUDA context's unique id (cuCtxGetId: ids are not reused within a
// process), or 0 if the driver cannot tell.  Per-context state the library caches
// (a module's symbol address, a kernel's shared-memory attribute) is keyed by it, so a
// new context (after cudaDeviceReset, or another context made current) is noticed.
// The two driver calls are looked up once through the runtime.
inline unsigned long long current_context_id()
{
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

inline kvl_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? KVL_OK : KVL_ECUDA;
}

}  // namespace kvl

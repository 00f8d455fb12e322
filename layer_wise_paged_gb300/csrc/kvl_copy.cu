// kvl_copy.cu -- the per-layer copy kernels of libkvl.so: slice, merge-scatter into
// the paged pool, and gather / scatter-back of per-layer K/V objects.
//
// Work unit: one work item of the plan, i.e. one logical block j of one request
// (Tutti 阅读笔记, 伪代码 1: retrieve_layer walks a layer's block ids; here every
// (request, block) of the batch is one item of a single launch per layer).  Its rows
// are the block's token slots of each plane (merge-scatter, gather, scatter-back) or
// the block's token rows of the layer (slice).
//
// A CTA is one warp driving the Tensor Memory Accelerator's bulk copies, on every
// SM of a persistent grid:
//   * scheduling: CTA b takes items b and b + G, then claims further items one at a
//     time from a per-(layer, op) counter in the plan (atomicAdd, issued one item
//     ahead), so faster SMs take more items and all finish together; every CTA stops
//     after its first claim past the end, so a launch's claims are counted in advance,
//     and the CTA that draws the last of them rewinds the counter for the next launch
//     (no CTA waits on an atomic on its way out);
//   * metadata: the plan resolved every item into a 128-byte record (bases and
//     strides at layer 0, pool block id, hit / valid slot counts); the warp loads the
//     next item's record (one word per lane) while the current item's copies run,
//     and reads fields from their lanes with shuffles;
//   * loads, completing on the stage's mbarrier: a segment of strided rows (a token's
//     plane is not adjacent to the next token's in the full-block source) is one tiled
//     `cp.async.bulk.tensor` load through the plan's tensor map of its source when it
//     is a whole segment or a block's tail drawn from one mapped source, else one
//     `cp.async.bulk` load per row; a contiguous source run (gather / scatter-back) is one `cp.async.bulk`
//     load per segment;
//   * stores: one `cp.async.bulk` shared -> global per segment (a segment is a run of
//     slots of one item and plane, at most one stage long, whose destination is
//     contiguous), in bulk groups; a stage is refilled only after its store has read
//     it (`cp.async.bulk.wait_group.read`).
// Loads run up to STAGES - 1 segments ahead of stores across item boundaries, so
// each SM keeps over 100 KiB in flight (one 6-stage CTA, or two 3-stage CTAs of
// consecutive launches side by side) with no registers holding data.  Every mbarrier
// wait is bounded by the global timer: past the limit the kernel records
// KVL_ETIMEOUT, waits (bounded again) for its copies in flight and returns.
//
// Ordering between launches: programmatic dependent launch.  A kernel waits for its
// predecessor (griddepcontrol.wait) before its first read and then lets its successor
// launch; or, when the caller declared the two independent
// (KVL_LAUNCH_OVERLAP_PREVIOUS), it lets its successor launch at once and waits just
// before it exits, so it still completes after its predecessor.  With a plan the
// caller declared complete (KVL_LAUNCH_PLAN_READY), a waiting kernel checks the plan,
// reads its first records, acquires its first tensor maps, prefetches its first
// source rows into L2 (cp.async.bulk.prefetch), and works out its segment geometry and
// its first unit's addresses before the wait.
#include <cstdint>

#include "kvl_internal.cuh"

namespace kvl {
namespace {

enum Op { OP_SLICE = 0, OP_MERGE = 1, OP_GATHER = 2, OP_SCATTER = 3 };

#ifndef KVL_PDL
#define KVL_PDL 1
#endif

// Pipeline depth.  A launch that has its SMs to itself keeps kDeepStages stages (192
// KiB): one CTA must keep enough bytes in flight to hold its SM's share of the HBM
// bandwidth.  A launch that may overlap the one before it (KVL_LAUNCH_OVERLAP_PREVIOUS),
// or that precedes one (KVL_LAUNCH_SHARE_SMS), keeps kShallowStages (96 KiB), so a CTA
// of each of two consecutive launches fits on one SM: while one launch drains its last
// items, the next one's CTAs already stream, and two CTAs per SM together keep as many
// bytes in flight as one deep CTA.
constexpr int kDeepStages = 6;
constexpr int kShallowStages = 3;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per mbarrier wait
static_assert(kStageBytes % 16 == 0 && kShallowStages >= 2 && kDeepStages >= kShallowStages,
              "stage geometry");

struct CopyArgs {
    void *plan;
    uint64_t plan_bytes;  // bytes of the caller's plan buffer: no plan read goes beyond
    const kvl_request *reqs;
    const int32_t *tables;
    uint8_t *pool;
    uint8_t *out;  // hit_out (slice), complete_out (merge, may be null)
    int32_t P, B, Rp, layer, L;
    int32_t layer_count;  // layers [layer, layer + layer_count) in this launch
    int32_t flags;        // KVL_LAUNCH_* of the call
    int64_t N;
};

// Per work item, the bases its rows are addressed from (see item_meta).
struct ItemMeta {
    const uint8_t *src_a;  // first source (hit rows / pool block / objects)
    const uint8_t *src_b;  // miss rows (merge)
    uint8_t *dst;          // destination base
    uint8_t *dst2;         // complete_layer rows (merge, optional)
    int64_t a_stride;      // bytes between source rows of src_a
    int64_t b_stride;      // bytes between source rows of src_b
    int64_t src_pstride;   // bytes between planes, source side
    int64_t dst_pstride;   // bytes between planes, destination side
    int32_t n_a;           // rows (slots) served by src_a
    int32_t n_valid;       // rows (slots) that exist
    // Tensor maps of the two sources, of whole segments and of block tails (null:
    // per-row loads), with the coordinates of slot 0 and the dim order of each source
    // (slice and merge-scatter only).
    const uint8_t *map_a, *map_a_tail, *map_b, *map_b_tail;
    int32_t blk_a, tok_a, tok_b;
    bool layer_first_a, layer_first_b;
};

// ---- PTX wrappers ----------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_inval(uint32_t bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for a phase of a stage's mbarrier; false when the limit passed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Complete `bytes` of an mbarrier's expected transaction count from this thread.
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void *src, uint32_t bytes,
                                          uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_smem),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// One box of a 5-D tensor map (coordinates innermost first) into shared memory,
// completing on the stage's mbarrier like bulk_load.
__device__ __forceinline__ void tensor_load_5d(uint32_t dst_smem, const void *map, int32_t c0,
                                               int32_t c1, int32_t c2, int32_t c3, int32_t c4,
                                               uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst_smem),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}

// The plan wrote its tensor maps with generic stores and a release to the tensor-map
// proxy; this is the matching acquire, before the first tensor load through `map`.
__device__ __forceinline__ void acquire_tensor_map(const void *map)
{
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, uint32_t src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(src_smem), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the newest store group have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_one()
{
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Programmatic dependent launch: the next kernel on the stream may be scheduled
// while this one runs; it waits for this grid's completion (and its memory) in
// grid_dependency_wait() before touching any data.
__device__ __forceinline__ void allow_dependents_launch()
{
#if KVL_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

__device__ __forceinline__ void grid_dependency_wait()
{
#if KVL_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

// Warm L2 with the line holding p.  A hint only: L2 is the device's point of
// coherence, so a line fetched before a preceding kernel's writes land is updated by
// them, and no later load can see it stale.
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2: a hint, with
// the same coherence as prefetch_l2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 32-bit load through the read-only path; volatile so that it is issued where it
// stands, ahead of the loads that follow it.
__device__ __forceinline__ uint32_t ld_nc_u32(const void *p)
{
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Ordinary SM accesses, for the side of a copy that lives in pinned host memory.
__device__ __forceinline__ uint4 ld_global_v4(const uint8_t *p)
{
    uint4 r;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_global_v4(uint8_t *p, const uint4 &v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t a)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(a));
    return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t a, const uint4 &v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Read `nrows` rows of `row_bytes` (row r at rowptr(r)) into shared memory at
// sbase + r*row_bytes with 16-byte loads: four rows and four vectors per lane, 8 KiB a
// warp, in flight per round trip (NVLink-C2C round trips take microseconds).
template <typename RowPtr>
__device__ __forceinline__ void lsu_rows_to_smem(const RowPtr &rowptr, int nrows, int row_bytes,
                                                 uint32_t sbase, int lane)
{
    constexpr int kRows = 4, kVec = 4;
    const int vpr = row_bytes >> 4;
    for (int r = 0; r < nrows; r += kRows) {
        const uint8_t *p[kRows];
#pragma unroll
        for (int q = 0; q < kRows; ++q) p[q] = r + q < nrows ? rowptr(r + q) : nullptr;
        for (int c0 = 0; c0 < vpr; c0 += 32 * kVec) {
            uint4 x[kRows][kVec];
#pragma unroll
            for (int q = 0; q < kRows; ++q)
#pragma unroll
                for (int k = 0; k < kVec; ++k) {
                    const int c = c0 + k * 32 + lane;
                    if (p[q] && c < vpr) x[q][k] = ld_global_v4(p[q] + c * 16);
                }
#pragma unroll
            for (int q = 0; q < kRows; ++q)
#pragma unroll
                for (int k = 0; k < kVec; ++k) {
                    const int c = c0 + k * 32 + lane;
                    if (p[q] && c < vpr)
                        st_shared_v4(sbase + uint32_t(r + q) * uint32_t(row_bytes) + uint32_t(c) * 16,
                                     x[q][k]);
                }
        }
    }
}

// Write `bytes` of shared memory at `src` to global `dst` with 16-byte stores.
__device__ __forceinline__ void lsu_smem_to_global(uint8_t *dst, uint32_t src, uint32_t bytes, int lane)
{
    for (uint32_t v = lane; v < bytes / 16; v += 32) st_global_v4(dst + v * 16, ld_shared_v4(src + v * 16));
}

template <typename T>
__device__ __forceinline__ T shfl_ptr(T p, int src)
{
    return reinterpret_cast<T>(__shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(p), src));
}

// ---- plan checks and metadata ------------------------------------------------

// A plan matches a call when it was built (magic) for this geometry, request array
// and block tables, and fits the caller's buffer with the request count it records;
// these header fields never change after the plan is built.  The checks keep every
// later index inside the plan's own arrays (all of them below plan_bytes) and the
// request array it was sized for.  The plan is usable when it also recorded no error
// (its status word, which copy calls may write).
template <int OP>
__device__ __forceinline__ bool plan_matches(const CopyArgs &a)
{
    PlanHeader *h = static_cast<PlanHeader *>(a.plan);
    const int32_t n_req = h->n_req;
    if (h->magic != kPlanMagic || h->pool_blocks != a.N || h->block_tokens != a.B ||
        h->n_layers != a.L || h->n_planes != a.P || h->plane_row_bytes != a.Rp ||
        h->reqs != a.reqs || (OP != OP_SLICE && h->tables != a.tables) || n_req < 0 ||
        plan_layout(n_req, a.N, a.L).off[8] > a.plan_bytes) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(h, KVL_EINVAL, 0);
        return false;
    }
    return true;
}

// Field of the item record held one word per lane.
__device__ __forceinline__ uint32_t rec_word(uint32_t rec, int w) { return __shfl_sync(0xffffffffu, rec, w); }

__device__ __forceinline__ uint64_t rec_u64(uint32_t rec, int w)
{
    return uint64_t(rec_word(rec, w)) | (uint64_t(rec_word(rec, w + 1)) << 32);
}

// The bases and strides the item's rows are copied through, for this op and layer,
// from the item's record.  False (after recording the error) when this op cannot
// copy the item.
template <int OP>
__device__ __forceinline__ bool item_meta(const CopyArgs &a, PlanHeader *h, const uint8_t *maps,
                                          uint32_t rec, int64_t l, int64_t n_hit_all,
                                          int64_t n_tok_all, ItemMeta &m)
{
    const int64_t B = a.B, Rp = a.Rp;
    const int64_t lo = l - a.layer;  // output layer within this launch
    const int64_t b = int32_t(rec_word(rec, 22));
    const int32_t n_hit = int32_t(rec_word(rec, 23));
    const int32_t n_valid = int32_t(rec_word(rec, 24));
    const int32_t req = int32_t(rec_word(rec, 25));
    const uint64_t hit_base = rec_u64(rec, 0), miss_base = rec_u64(rec, 6), obj_base = rec_u64(rec, 12);
    const int64_t hit_ts = int64_t(rec_u64(rec, 2)), hit_ls = int64_t(rec_u64(rec, 4));
    const int64_t miss_ts = int64_t(rec_u64(rec, 8)), miss_ls = int64_t(rec_u64(rec, 10));
    const int64_t obj_ps = int64_t(rec_u64(rec, 14)), obj_ls = int64_t(rec_u64(rec, 16));
    const int64_t hit_row = int64_t(rec_u64(rec, 18)), tok_row = int64_t(rec_u64(rec, 20));
    const int64_t R = int64_t(a.P) * Rp;
    m.src_a = reinterpret_cast<const uint8_t *>(hit_base + uint64_t(l * hit_ls));
    m.src_b = reinterpret_cast<const uint8_t *>(miss_base + uint64_t(l * miss_ls));
    m.a_stride = hit_ts;
    m.b_stride = miss_ts;
    m.n_a = n_hit;
    m.n_valid = n_valid;
    m.dst2 = nullptr;
    m.map_a = m.map_a_tail = m.map_b = m.map_b_tail = nullptr;
    if (maps && (OP == OP_SLICE || OP == OP_MERGE)) {
        const int32_t flags = int32_t(rec_word(rec, 29));
        const uint8_t *req_maps = maps + int64_t(req) * (kMapsPerReq * kMapBytes);
        auto map_of = [&](int k) { return (flags & map_bit(k)) ? req_maps + k * kMapBytes : nullptr; };
        const int hit_kind = OP == OP_SLICE ? MAP_SLICE : MAP_HIT;
        m.map_a = map_of(hit_kind);
        m.map_a_tail = map_of(hit_kind + kMapTail);
        if (OP == OP_MERGE) {
            m.map_b = map_of(MAP_MISS);
            m.map_b_tail = map_of(MAP_MISS_TAIL);
        }
        m.blk_a = int32_t(rec_word(rec, 26));
        m.tok_a = int32_t(rec_word(rec, 27));
        m.tok_b = int32_t(rec_word(rec, 28));
        m.layer_first_a = (flags & kMapHitLayerFirst) != 0;
        m.layer_first_b = (flags & kMapMissLayerFirst) != 0;
    }
    uint8_t *pool_blk = a.pool + ((l * a.P) * a.N + b) * B * Rp;
    const int64_t pool_ps = a.N * B * Rp;
    if (OP == OP_SLICE) {
        m.n_valid = n_hit;
        m.src_pstride = 0;
        m.dst = a.out + (lo * n_hit_all + hit_row) * R;
        m.dst_pstride = 0;
        return true;
    }
    if (OP == OP_MERGE) {
        m.src_pstride = Rp;
        m.dst = pool_blk;
        m.dst_pstride = pool_ps;
        if (a.out) m.dst2 = a.out + (lo * n_tok_all + tok_row) * R;
        return true;
    }
    if (obj_base == 0) {
        if ((threadIdx.x & 31) == 0) record_error(h, KVL_EINVAL, (unsigned long long)req);
        return false;
    }
    uint8_t *obj = reinterpret_cast<uint8_t *>(obj_base + uint64_t(l * obj_ls));
    m.n_a = m.n_valid = int32_t(B);  // objects carry whole blocks
    m.a_stride = Rp;
    if (OP == OP_GATHER) {
        m.src_a = pool_blk;
        m.src_pstride = pool_ps;
        m.dst = obj;
        m.dst_pstride = obj_ps;
    } else {
        m.src_a = obj;
        m.src_pstride = obj_ps;
        m.dst = pool_blk;
        m.dst_pstride = pool_ps;
    }
    return true;
}

// grid_dependency_wait with the fields of `m` and the segment geometry the first
// copies use as operands, so that they are computed before the wait rather than
// after it.
__device__ __forceinline__ void grid_dependency_wait_after(const ItemMeta &m, int max_rows,
                                                           int box_rows, int tail_rows,
                                                           int plane_chunks)
{
#if KVL_PDL
    asm volatile("griddepcontrol.wait;" ::"l"(m.src_a), "l"(m.src_b), "l"(m.dst), "l"(m.map_a),
                 "l"(m.a_stride), "l"(m.dst_pstride), "r"(m.n_valid), "r"(m.n_a), "r"(m.tok_a),
                 "r"(m.blk_a), "r"(max_rows), "r"(box_rows), "r"(tail_rows), "r"(plane_chunks)
                 : "memory");
#endif
}

// Prefetch into L2 the source bytes unit (rec, layer l) will read first, at most
// `budget` of them; returns the bytes asked for.  Token rows of the slice and
// merge-scatter (a row's P planes are adjacent in both sources: R bytes), whole
// plane-blocks of the gather and scatter-back.  Reads only the item record, which the
// plan resolved from addresses its requests declare.
template <int OP>
__device__ __forceinline__ uint32_t prefetch_unit(const CopyArgs &a, uint32_t rec, int64_t l,
                                                  uint32_t budget, int lane)
{
    const int64_t Rp = a.Rp, R = int64_t(a.P) * Rp;
    if (OP == OP_SLICE || OP == OP_MERGE) {
        // all fields first, by the whole warp (shuffles), then the lane-divergent loop
        const int32_t n_hit = int32_t(rec_word(rec, 23));
        const int32_t n = OP == OP_SLICE ? n_hit : int32_t(rec_word(rec, 24));
        const uint64_t hit = rec_u64(rec, 0) + uint64_t(l * int64_t(rec_u64(rec, 4)));
        const uint64_t miss = rec_u64(rec, 6) + uint64_t(l * int64_t(rec_u64(rec, 10)));
        const int64_t hit_ts = int64_t(rec_u64(rec, 2)), miss_ts = int64_t(rec_u64(rec, 8));
        const int32_t rows = int32_t(int64_t(n) < int64_t(budget) / R ? int64_t(n) : int64_t(budget) / R);
        for (int s = lane; s < rows; s += 32) {
            const uint64_t src = s < n_hit ? hit + uint64_t(s * hit_ts) : miss + uint64_t(s * miss_ts);
            bulk_prefetch_l2(reinterpret_cast<const void *>(src), uint32_t(R));
        }
        return uint32_t(rows * R);
    }
    // every field is read here, by the whole warp: the shuffles must not sit inside the
    // lane-divergent loop below
    const uint64_t obj = rec_u64(rec, 12);
    const int64_t obj_ps = int64_t(rec_u64(rec, 14)), obj_ls = int64_t(rec_u64(rec, 16));
    const int64_t b = int32_t(rec_word(rec, 22));
    const int64_t blk = int64_t(a.B) * Rp;
    const int32_t planes = int32_t(int64_t(a.P) < int64_t(budget) / blk ? int64_t(a.P) : int64_t(budget) / blk);
    if (obj == 0) return budget;  // the copy itself records the missing objects
    for (int p = lane; p < planes; p += 32) {
        const uint8_t *src = OP == OP_GATHER
            ? a.pool + ((l * a.P + p) * a.N + b) * blk
            : reinterpret_cast<const uint8_t *>(obj + uint64_t(l * obj_ls + p * obj_ps));
        bulk_prefetch_l2(src, uint32_t(blk));
    }
    return uint32_t(planes * blk);
}

// ---- the pipelined copy --------------------------------------------------------

struct StageInfo {
    uint8_t *dst;       // contiguous destination of the segment
    uint8_t *dst2;      // complete_layer row of the segment's first slot (or null)
    uint32_t bytes;     // segment bytes (= rows * row_bytes)
    uint32_t rows;
};

// HOST: 0 = every buffer in device memory (bulk copies both ways), 1 = sources in
// pinned host memory (SM loads), 2 = destinations in pinned host memory (SM stores).
template <int OP, int HOST, int STAGES>
__device__ __forceinline__ void copy_rows(const CopyArgs &a)
{
    constexpr int kStages = STAGES;
    constexpr int kLookahead = kStages - 1;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kStages];
    __shared__ StageInfo info[kStages];

    const int lane = threadIdx.x;
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    // The item records sit at a fixed offset, so this CTA's first record (item
    // blockIdx.x, below the plan's capacity of N records, which the host has checked
    // lie inside plan_bytes) is addressed without the header.  Its line and the
    // header's are fetched into L2 while the previous kernel drains, and read together
    // once it has finished.
    const uint8_t *plan_base = static_cast<const uint8_t *>(a.plan);
    const bool first_in_cap = blockIdx.x < a.N;
    const uint32_t *first_rec = reinterpret_cast<const uint32_t *>(
        plan_base + kRecordsOffset + int64_t(blockIdx.x) * int64_t(sizeof(ItemRec)));
    if (lane == 0) prefetch_l2(plan_base);
    if (lane == 1 && first_in_cap) prefetch_l2(first_rec);
    __syncwarp();
    // Everything this kernel reads may come from the previous kernel on the stream,
    // unless the caller declared the two independent: then the wait moves to the end,
    // so this kernel still completes after the previous one.  With a plan the caller
    // declared complete (KVL_LAUNCH_PLAN_READY), the plan is checked and the first
    // units' source rows are prefetched into L2 before the wait.
    const bool overlap = (a.flags & KVL_LAUNCH_OVERLAP_PREVIOUS) != 0;
    const bool early = HOST == 0 && !overlap && (a.flags & KVL_LAUNCH_PLAN_READY) != 0;
    if (!overlap && !early) grid_dependency_wait();
    // Dependents are let go only once this kernel has passed its own wait (or, when it
    // overlaps its predecessor, at once): a later launch that overlaps this one must
    // not start before the kernels this one waits for have finished.
    if (!early) allow_dependents_launch();
    const uint32_t rec_first = first_in_cap ? ld_nc_u32(first_rec + lane) : 0u;
    bool usable = plan_matches<OP>(a);
    // The header fields below never change once the plan is built.  A launch with a
    // complete plan (early) reads them, and acquires the tensor maps its first unit
    // reads through, before its dependency wait, so that after the wait only the
    // status word stands between it and its first load.
    PlanHeader *h = static_cast<PlanHeader *>(a.plan);
    PlanView v;
    int64_t n_items = 0, n_hit_all = 0, n_tok_all = 0;
    int32_t map_chunk = 0;
    constexpr bool kMaps = HOST == 0 && (OP == OP_SLICE || OP == OP_MERGE);
    // Segment geometry, from the call's arguments (and, for the tensor maps' chunks,
    // the header): worked out before the dependency wait when the plan is complete.
    const int planes = OP == OP_SLICE ? 1 : a.P;
    const int row_bytes = OP == OP_SLICE ? a.P * a.Rp : a.Rp;
    const int max_rows = kStageBytes / row_bytes;  // >= 1 (host-checked)
    const int64_t R = int64_t(a.P) * a.Rp;
    const int box_rows = segment_rows(a.B, row_bytes);        // a whole segment's box
    const int tail_rows = segment_tail_rows(a.B, row_bytes);  // a block tail's box (0: none)
    int32_t plane_chunks = 0;
    auto read_header = [&]() {
        v = plan_view(a.plan, h->n_req, h->pool_blocks, h->n_layers);
        n_items = h->n_items;
        n_hit_all = h->n_hit;
        n_tok_all = h->n_tokens;
        map_chunk = kMaps ? h->map_chunk : 0;
        plane_chunks = map_chunk > 0 ? a.Rp / map_chunk : 0;
    };
    // lane 0's four most recently acquired maps, newest first
    const uint8_t *acq0 = nullptr, *acq1 = nullptr, *acq2 = nullptr, *acq3 = nullptr;
    bool header_read = false;
    // the first unit's addresses, worked out before the wait by a launch with a
    // complete plan (decoding a record takes a few hundred cycles of one warp)
    ItemMeta m_first = {};
    bool m_first_ready = false, m_first_ok = false;
    if (early) {
        // The plan was complete before the previous kernel began: a status of OK now
        // means every item record was written, and the records never change after.
        if (usable && h->status == KVL_OK) {
            read_header();
            header_read = true;
            const int64_t n_units = n_items * a.layer_count;
            uint32_t budget = uint32_t(kStages) * uint32_t(kStageBytes);
            // this CTA's two statically placed units, as far as the pipeline holds
            for (int k = 0; k < 2 && budget > 0; ++k) {
                const int64_t u = int64_t(blockIdx.x) + int64_t(k) * gridDim.x;
                if (u >= n_units) break;
                const int64_t item = u % n_items;
                const uint32_t rec = u < n_items ? rec_first
                    : ld_nc_u32(reinterpret_cast<const uint32_t *>(
                                    plan_base + kRecordsOffset + item * int64_t(sizeof(ItemRec))) + lane);
                budget -= prefetch_unit<OP>(a, rec, a.layer + u / n_items, budget, lane);
            }
            // the tensor maps of the first unit's request that this op reads through
            // (at most four: a kind and its tail kind for each of two sources)
            if (kMaps && map_chunk > 0 && int64_t(blockIdx.x) < n_items) {
                const int32_t flags = int32_t(rec_word(rec_first, 29));
                const uint8_t *req_maps = v.maps + int64_t(int32_t(rec_word(rec_first, 25))) *
                                                       (kMapsPerReq * kMapBytes);
                if (lane == 0) {
                    const int kinds[4] = {OP == OP_SLICE ? MAP_SLICE : MAP_HIT,
                                          (OP == OP_SLICE ? MAP_SLICE : MAP_HIT) + kMapTail,
                                          OP == OP_SLICE ? -1 : MAP_MISS,
                                          OP == OP_SLICE ? -1 : MAP_MISS + kMapTail};
                    for (int i = 0; i < 4; ++i) {
                        if (kinds[i] < 0 || !(flags & map_bit(kinds[i]))) continue;
                        const uint8_t *m = req_maps + kinds[i] * kMapBytes;
                        acquire_tensor_map(m);
                        acq3 = acq2;
                        acq2 = acq1;
                        acq1 = acq0;
                        acq0 = m;
                    }
                }
            }
            if (int64_t(blockIdx.x) < n_items) {  // unit blockIdx.x: item blockIdx.x, first layer
                m_first_ok = item_meta<OP>(a, h, map_chunk > 0 ? v.maps : nullptr, rec_first,
                                           a.layer, n_hit_all, n_tok_all, m_first);
                m_first_ready = true;
            }
        }
        grid_dependency_wait_after(m_first, max_rows, box_rows, tail_rows, plane_chunks);
        allow_dependents_launch();
    }
    usable = usable && h->status == KVL_OK;
    if (!usable) {
        if (lane == 0)
            for (int s = 0; s < kStages; ++s) mbar_inval(bar0 + 8 * s);
        if (overlap) grid_dependency_wait();
        return;
    }
    if (!header_read) read_header();
    ClaimCounter *ctr = &v.counters[int64_t(a.layer) * kOps + OP];
    const int64_t G = gridDim.x;

    // Tensor maps (device buffers only): a segment of box_rows rows from one source
    // that has a map is one tensor load; plane p starts at chunk p * Rp / chunk.
    const uint8_t *maps = map_chunk > 0 ? v.maps : nullptr;

    int64_t issued = 0, retired = 0;
    bool timed_out = false;
    constexpr bool host_src = HOST == 1;
    constexpr bool host_dst = HOST == 2;

    // Retire the oldest issued segment: wait for its loads, store it.
    auto retire = [&]() {
        const int st = int(retired % kStages);
        const uint32_t parity = uint32_t((retired / kStages) & 1);
        // warp-uniform verdict: every lane polls, all must have seen the phase
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * st, parity))) {
            timed_out = true;
            return;
        }
        fence_proxy_async_smem();
        const StageInfo si = info[st];
        const uint32_t src = smem0 + uint32_t(st) * kStageBytes;
        if constexpr (host_dst) {
            // the destination is host memory: SM stores over NVLink-C2C
            if (OP == OP_MERGE && si.dst2 != nullptr)
                for (uint32_t i = 0; i < si.rows; ++i)
                    lsu_smem_to_global(si.dst2 + int64_t(i) * R, src + i * uint32_t(row_bytes),
                                       uint32_t(row_bytes), lane);
            lsu_smem_to_global(si.dst, src, si.bytes, lane);
            // the stage's generic reads come before the next bulk load into it
            fence_proxy_async_smem();
            __syncwarp();
        } else {
            if (OP == OP_MERGE && si.dst2 != nullptr) {
                for (uint32_t i = lane; i < si.rows; i += 32)
                    bulk_store(si.dst2 + int64_t(i) * R, src + i * uint32_t(row_bytes), uint32_t(row_bytes));
            }
            if (lane == 0) bulk_store(si.dst, src, si.bytes);
        }
        bulk_commit();
        ++retired;
    };

    auto load_rec = [&](int64_t item) -> uint32_t {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(v.items + item);
        return __ldg(w + lane);
    };

    // Work units: (layer, item) pairs, layer by layer, over the launch's layers.  CTA b
    // takes units b and b + G; later units are claimed from the counter (its values
    // count from the 2G statically placed units), one claim in flight ahead, and never
    // waited on before it is needed.  An item's planes are copied back to back by one
    // CTA: for the slice and merge-scatter they are the two halves of the same source
    // token rows, which DRAM serves best close together in time.
    // unit u = (layer a.layer + u / n_items, item u % n_items); the host keeps
    // n_units < 2^31, so 32-bit arithmetic suffices, and a one-layer launch divides
    // nothing
    const int64_t n_units = n_items * a.layer_count;
    const uint32_t n_items32 = uint32_t(n_items);
    const bool one_layer = a.layer_count == 1;
    auto item_of = [&](int64_t u) -> int64_t { return one_layer ? u : int64_t(uint32_t(u) % n_items32); };
    auto layer_of = [&](int64_t u) -> int64_t {
        return int64_t(a.layer) + (one_layer ? 0 : int64_t(uint32_t(u) / n_items32));
    };
    int64_t cur = blockIdx.x;
    const int64_t nxt_static = blockIdx.x + G;
    // unit cur < n_items is item cur of the first layer: the record read above
    uint32_t rec_cur = cur < n_items ? rec_first : cur < n_units ? load_rec(item_of(cur)) : 0u;
    // Every CTA claims until its first claim past the last unit and then stops, so a
    // launch draws exactly max(n_units - 2G, 0) + G claims, numbered from 0.  The CTA
    // that reads the last of them rewinds the counter for the next launch on it: no
    // claim of this launch can follow.  (A launch in which some CTA stops early, on a
    // timeout or on a plan status that turned to an error, may leave the counter
    // unrewound; its plan then carries that error, which makes every later copy call
    // on it a no-op until the plan is rebuilt, and a rebuild clears the counters.)
    // A CTA draws its first claim once its first load is on its way (or when it has no
    // load to issue): every CTA of a launch draws it at about the same moment, so the
    // atomics queue at the counter, and nothing before the first load waits for one.
    const uint32_t last_claim = uint32_t((n_units > 2 * G ? n_units - 2 * G : 0) + G - 1);
    uint32_t claim = 0;
    bool claim_unread = false, first_claim_due = true;
    auto draw_claim = [&]() {
        if (lane == 0) claim = atomicAdd(&ctr->next, 1u);
        claim_unread = true;
        first_claim_due = false;
    };
    auto read_claim = [&]() -> uint32_t {
        const uint32_t c = __shfl_sync(0xffffffffu, claim, 0);
        if (claim_unread && c == last_claim && lane == 0) atomicExch(&ctr->next, 0u);
        claim_unread = false;
        return c;
    };
    for (bool first = true;; first = false) {
        int64_t nxt;
        if (first) {
            nxt = nxt_static;
        } else {
            if (first_claim_due) draw_claim();  // the first unit issued no load
            nxt = 2 * G + int64_t(read_claim());
            if (nxt < n_units) draw_claim();
        }
        uint32_t rec_nxt = 0;
        if (nxt < n_units) rec_nxt = load_rec(item_of(nxt));
        if (cur >= n_units || timed_out) break;

        ItemMeta m;
        const int64_t l_cur = layer_of(cur);
        bool meta_ok;
        if (first && m_first_ready) {
            m = m_first;
            meta_ok = m_first_ok;
        } else {
            meta_ok = item_meta<OP>(a, h, maps, rec_cur, l_cur, n_hit_all, n_tok_all, m);
        }
        if (meta_ok) {
          for (int p = 0; p < planes && !timed_out; ++p) {
            for (int s0 = 0; s0 < m.n_valid && !timed_out; s0 += max_rows) {
                const int ns = m.n_valid - s0 < max_rows ? m.n_valid - s0 : max_rows;
                // make room: keep at most kLookahead segments in flight
                if (issued - retired >= kLookahead) {
                    retire();
                    if (timed_out) break;
                }
                const int st = int(issued % kStages);
                if (issued >= kStages) bulk_wait_read_all_but_one();
                const uint32_t sbase = smem0 + uint32_t(st) * kStageBytes;
                const uint32_t bar = bar0 + 8 * st;
                const uint32_t bytes = uint32_t(ns) * uint32_t(row_bytes);
                if (lane == 0) {
                    StageInfo si;
                    si.dst = m.dst + p * m.dst_pstride + int64_t(s0) * row_bytes;
                    si.dst2 = (OP == OP_MERGE && m.dst2) ? m.dst2 + int64_t(s0) * R + int64_t(p) * a.Rp
                                                         : nullptr;
                    si.bytes = bytes;
                    si.rows = uint32_t(ns);
                    info[st] = si;
                    if (!host_src) mbar_arrive_expect_tx(bar, bytes);
                }
                __syncwarp();
                if constexpr (host_src) {
                    // the source is host memory: SM loads over NVLink-C2C into the stage
                    if (OP == OP_GATHER || OP == OP_SCATTER) {
                        const uint8_t *base = m.src_a + p * m.src_pstride + int64_t(s0) * row_bytes;
                        lsu_rows_to_smem([&](int i) { return base + int64_t(i) * row_bytes; }, ns,
                                         row_bytes, sbase, lane);
                    } else {
                        lsu_rows_to_smem(
                            [&](int i) {
                                const int64_t s = s0 + i;
                                return (s < m.n_a ? m.src_a + s * m.a_stride : m.src_b + s * m.b_stride) +
                                       int64_t(p) * m.src_pstride;
                            },
                            ns, row_bytes, sbase, lane);
                    }
                    // the stage's generic writes come before the bulk store that reads it
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar);
                } else if (OP == OP_GATHER || OP == OP_SCATTER) {
                    if (lane == 0)
                        bulk_load(sbase, m.src_a + p * m.src_pstride + int64_t(s0) * row_bytes, bytes, bar);
                } else if (const uint8_t *map = !kMaps ? nullptr
                                                : ns == box_rows
                                                    ? (s0 + ns <= m.n_a ? m.map_a : s0 >= m.n_a ? m.map_b : nullptr)
                                                : ns == tail_rows
                                                    ? (s0 + ns <= m.n_a ? m.map_a_tail
                                                       : s0 >= m.n_a   ? m.map_b_tail
                                                                       : nullptr)
                                                    : nullptr) {
                    // a whole segment or a block tail from one mapped source: one box
                    if (lane == 0) {
                        if (map != acq0 && map != acq1 && map != acq2 && map != acq3) {
                            acquire_tensor_map(map);
                            acq3 = acq2;
                            acq2 = acq1;
                            acq1 = acq0;
                            acq0 = map;
                        }
                        const bool from_a = s0 + ns <= m.n_a;
                        const int32_t tok = (from_a ? m.tok_a : m.tok_b) + s0;
                        const int32_t lay = int32_t(l_cur);
                        const bool lf = from_a ? m.layer_first_a : m.layer_first_b;
                        tensor_load_5d(sbase, map, 0, OP == OP_MERGE ? p * plane_chunks : 0,
                                       lf ? lay : tok, lf ? tok : lay, from_a ? m.blk_a : 0, bar);
                    }
                } else {
                    for (int i = lane; i < ns; i += 32) {
                        const int64_t s = s0 + i;
                        const uint8_t *src = s < m.n_a ? m.src_a + s * m.a_stride
                                                       : m.src_b + s * m.b_stride;
                        bulk_load(sbase + uint32_t(i) * uint32_t(row_bytes),
                                  src + int64_t(p) * m.src_pstride, uint32_t(row_bytes), bar);
                    }
                }
                ++issued;
                if (first_claim_due) draw_claim();
            }
          }
        }
        cur = nxt;
        rec_cur = rec_nxt;
    }
    while (retired < issued && !timed_out) retire();
    // a CTA with no unit of its own still draws its claim, and every CTA reads its last
    if (first_claim_due) draw_claim();
    if (claim_unread) read_claim();

    if (timed_out) {
        if (lane == 0) record_error(h, KVL_ETIMEOUT, (unsigned long long)blockIdx.x);
        // let the loads still in flight land (bounded) before the CTA leaves
        for (int64_t k = retired; k < issued; ++k)
            mbar_wait_bounded(bar0 + 8 * int(k % kStages), uint32_t((k / kStages) & 1));
    }
    bulk_wait_all();
    __syncwarp();
    if (lane == 0)
        for (int s = 0; s < kStages; ++s) mbar_inval(bar0 + 8 * s);
    if (overlap) grid_dependency_wait();
}

// Diagnostic: the copy kernels' bounded wait, made to run out.  The barrier expects
// 16 bytes that no copy will deliver; after limit_ns the wait gives up and the kernel
// records KVL_ETIMEOUT, then completes the 16 bytes itself so the barrier's phase ends
// and it can be invalidated.  No memory is copied, nothing is left in flight.
__global__ void __launch_bounds__(32) kvl_wait_timeout_kernel(int32_t *status,
                                                              unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(b, 16);
    }
    __syncwarp();
    const bool done = __all_sync(0xffffffffu, mbar_wait_bounded(b, 0, limit_ns));
    if (threadIdx.x == 0) {
        *status = done ? KVL_OK : KVL_ETIMEOUT;
        if (!done) mbar_complete_tx(b, 16);
    }
    __syncwarp();
    mbar_wait_bounded(b, 0, limit_ns);
    __syncwarp();
    if (threadIdx.x == 0) mbar_inval(b);
}

// One kernel per op for device buffers, so launch lists and profiles name the op, in
// the two pipeline depths; the host-memory variants are separate instantiations (deep
// only: their SM loads or stores, not the stage count, set their pace), so the device
// path carries none of their code.
template <int STAGES>
__global__ void __launch_bounds__(32) kvl_slice_kernel(CopyArgs a) { copy_rows<OP_SLICE, 0, STAGES>(a); }
template <int STAGES>
__global__ void __launch_bounds__(32) kvl_merge_scatter_kernel(CopyArgs a) { copy_rows<OP_MERGE, 0, STAGES>(a); }
template <int STAGES>
__global__ void __launch_bounds__(32) kvl_gather_kernel(CopyArgs a) { copy_rows<OP_GATHER, 0, STAGES>(a); }
template <int STAGES>
__global__ void __launch_bounds__(32) kvl_scatter_back_kernel(CopyArgs a) { copy_rows<OP_SCATTER, 0, STAGES>(a); }

template <int OP, int HOST>
__global__ void __launch_bounds__(32) kvl_host_copy_kernel(CopyArgs a)
{
    copy_rows<OP, HOST, kDeepStages>(a);
}

template <int OP, int HOST, int STAGES>
constexpr void (*kernel_of())(CopyArgs)
{
    if constexpr (HOST != 0) {
        return kvl_host_copy_kernel<OP, HOST>;
    } else {
        return OP == OP_SLICE ? kvl_slice_kernel<STAGES>
             : OP == OP_MERGE ? kvl_merge_scatter_kernel<STAGES>
             : OP == OP_GATHER ? kvl_gather_kernel<STAGES>
                               : kvl_scatter_back_kernel<STAGES>;
    }
}

// Grid: one CTA on every SM (or the caller's cap).  Opts each kernel into its shared
// memory once per context: the attribute belongs to the context, so it is set again
// when the device's current context has changed (after cudaDeviceReset, say); with no
// context id to compare, on every call.  Concurrent first calls may both set it.
template <int OP, int HOST, int STAGES>
int grid_size(const kvl_launch *opts)
{
    static std::atomic<unsigned long long> ready_ctx[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    const unsigned long long ctx = current_context_id();
    if (ctx == 0 || ready_ctx[dev].load(std::memory_order_acquire) != ctx) {
        if (cudaFuncSetAttribute(kernel_of<OP, HOST, STAGES>(),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 STAGES * kStageBytes) != cudaSuccess)
            return 0;
        ready_ctx[dev].store(ctx, std::memory_order_release);
    }
    const int full = sm_count();
    if (opts && opts->max_ctas > 0 && opts->max_ctas < full) return opts->max_ctas;
    return full;
}

template <int OP, int HOST, int STAGES>
kvl_status launch_mode(const CopyArgs &a, const kvl_launch *opts, void *stream)
{
    constexpr int kSmemBytes = STAGES * kStageBytes;
    const int grid = grid_size<OP, HOST, STAGES>(opts);
    if (grid <= 0) return KVL_ECUDA;
#if KVL_PDL
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel_of<OP, HOST, STAGES>(), a) != cudaSuccess) return KVL_ECUDA;
    return KVL_OK;
#else
    kernel_of<OP, HOST, STAGES>()<<<grid, 32, kSmemBytes, static_cast<cudaStream_t>(stream)>>>(a);
    return launch_status();
#endif
}

template <int OP>
kvl_status launch(const CopyArgs &args, const kvl_launch *opts, void *stream)
{
    CopyArgs a = args;
    a.flags = opts ? opts->flags : 0;
    const int32_t host = a.flags & (KVL_LAUNCH_HOST_SRC | KVL_LAUNCH_HOST_DST);
    if (host == KVL_LAUNCH_HOST_SRC) return launch_mode<OP, 1, kDeepStages>(a, opts, stream);
    if (host == KVL_LAUNCH_HOST_DST) return launch_mode<OP, 2, kDeepStages>(a, opts, stream);
    if (a.flags & (KVL_LAUNCH_OVERLAP_PREVIOUS | KVL_LAUNCH_SHARE_SMS))
        return launch_mode<OP, 0, kShallowStages>(a, opts, stream);
    return launch_mode<OP, 0, kDeepStages>(a, opts, stream);
}

kvl_status common_checks(const kvl_geom *g, const void *d_plan, size_t plan_bytes,
                         const kvl_request *d_reqs, int32_t layer, int32_t layer_count,
                         int32_t row_bytes, const kvl_launch *opts)
{
    const kvl_status s = check_geom(g);
    if (s) return s;
    constexpr int32_t kHostBoth = KVL_LAUNCH_HOST_SRC | KVL_LAUNCH_HOST_DST;
    constexpr int32_t kKnown = kHostBoth | KVL_LAUNCH_OVERLAP_PREVIOUS | KVL_LAUNCH_SHARE_SMS |
                               KVL_LAUNCH_PLAN_READY;
    if (opts && (opts->max_ctas < 0 || (opts->flags & ~kKnown) ||
                 (opts->flags & kHostBoth) == kHostBoth))
        return KVL_EINVAL;
    // d_reqs may be NULL (a plan of no requests); the device compares it with the
    // plan's own record of the array it was built from
    if (!d_plan) return KVL_EINVAL;
    if (!aligned16(d_plan) || !aligned16(d_reqs)) return KVL_EALIGN;
    // the smallest plan of this geometry (header, N item records, work list, claim
    // counters): every plan read a kernel makes before it has checked the header lies
    // below it
    if (plan_bytes < plan_layout(0, g->pool_blocks, g->n_layers).off[8]) return KVL_EINVAL;
    if (layer < 0 || layer_count < 1 || layer >= g->n_layers || layer_count > g->n_layers - layer)
        return KVL_EINVAL;
    if (g->pool_blocks * int64_t(layer_count) >= (int64_t(1) << 31)) return KVL_EINVAL;  // unit ids
    if (row_bytes > kStageBytes) return KVL_EINVAL;  // a row must fit one stage
    return KVL_OK;
}

CopyArgs make_args(const kvl_geom *g, const void *d_plan, size_t plan_bytes,
                   const kvl_request *d_reqs, const int32_t *tables, int32_t layer,
                   int32_t layer_count, void *pool, void *out)
{
    CopyArgs a;
    a.plan = const_cast<void *>(d_plan);
    a.plan_bytes = plan_bytes;
    a.reqs = d_reqs;
    a.tables = tables;
    a.pool = static_cast<uint8_t *>(pool);
    a.out = static_cast<uint8_t *>(out);
    a.P = g->n_planes;
    a.B = g->block_tokens;
    a.Rp = g->plane_row_bytes;
    a.layer = layer;
    a.layer_count = layer_count;
    a.flags = 0;
    a.L = g->n_layers;
    a.N = g->pool_blocks;
    return a;
}

}  // namespace
}  // namespace kvl

using namespace kvl;

extern "C" kvl_status kvl_slice_layer(const kvl_geom *geom, const void *d_plan, size_t plan_bytes,
                                      const kvl_request *d_reqs, int32_t layer, int32_t layer_count,
                                      void *d_hit_out, const kvl_launch *opts, void *stream)
{
    const int32_t rb = geom ? geom->n_planes * geom->plane_row_bytes : 0;
    kvl_status s = common_checks(geom, d_plan, plan_bytes, d_reqs, layer, layer_count, rb, opts);
    if (s) return s;
    if (!d_hit_out) return KVL_EINVAL;
    if (!aligned16(d_hit_out)) return KVL_EALIGN;
    return launch<OP_SLICE>(make_args(geom, d_plan, plan_bytes, d_reqs, nullptr, layer, layer_count,
                                      nullptr, d_hit_out),
                            opts, stream);
}

extern "C" kvl_status kvl_merge_scatter_paged(const kvl_geom *geom, const void *d_plan,
                                              size_t plan_bytes, const kvl_request *d_reqs,
                                              const int32_t *d_block_tables, int32_t layer,
                                              int32_t layer_count, void *d_pool,
                                              void *d_complete_out, const kvl_launch *opts,
                                              void *stream)
{
    kvl_status s = common_checks(geom, d_plan, plan_bytes, d_reqs, layer, layer_count,
                                 geom ? geom->plane_row_bytes : 0, opts);
    if (s) return s;
    if (!d_pool) return KVL_EINVAL;  // d_block_tables: as d_reqs
    if ((reinterpret_cast<uintptr_t>(d_block_tables) & 3u) || !aligned16(d_pool) ||
        (d_complete_out && !aligned16(d_complete_out)))
        return KVL_EALIGN;
    return launch<OP_MERGE>(make_args(geom, d_plan, plan_bytes, d_reqs, d_block_tables, layer,
                                      layer_count, d_pool, d_complete_out),
                            opts, stream);
}

extern "C" kvl_status kvl_gather_layer_objects(const kvl_geom *geom, const void *d_plan,
                                               size_t plan_bytes, const kvl_request *d_reqs,
                                               const int32_t *d_block_tables, int32_t layer,
                                               int32_t layer_count, void *d_pool, int32_t direction,
                                               const kvl_launch *opts, void *stream)
{
    kvl_status s = common_checks(geom, d_plan, plan_bytes, d_reqs, layer, layer_count,
                                 geom ? geom->plane_row_bytes : 0, opts);
    if (s) return s;
    if (!d_pool) return KVL_EINVAL;  // d_block_tables: as d_reqs
    if (direction != KVL_GATHER && direction != KVL_SCATTER_BACK) return KVL_EINVAL;
    if ((reinterpret_cast<uintptr_t>(d_block_tables) & 3u) || !aligned16(d_pool)) return KVL_EALIGN;
    const CopyArgs a = make_args(geom, d_plan, plan_bytes, d_reqs, d_block_tables, layer,
                                 layer_count, d_pool, nullptr);
    return direction == KVL_GATHER ? launch<OP_GATHER>(a, opts, stream)
                                   : launch<OP_SCATTER>(a, opts, stream);
}

extern "C" kvl_status kvl_diag_wait_timeout(int32_t limit_us, int32_t *d_status, void *stream)
{
    if (!d_status || limit_us < 1 || limit_us > 10000000) return KVL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_status) & 3u) return KVL_EALIGN;
    kvl_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        d_status, static_cast<unsigned long long>(limit_us) * 1000ull);
    return launch_status();
}

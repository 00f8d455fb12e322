// kvl_copy.cu -- the per-layer copy kernels of libkvl.so: slice, merge-scatter into
// the paged pool, and gather / scatter-back of per-layer K/V objects.
//
// Every op is a set of "rows": Rp-byte plane rows (merge-scatter, gather,
// scatter-back) or R-byte token rows (slice).  The rows of all work items of the
// plan form one flat row space; each warp of a persistent grid takes one
// contiguous, equal share of it (so work is balanced to within one row whatever the
// request mix), decodes (item -> request, block -> table entry -> addresses) per row
// and moves the row with 16-byte vector loads and stores, two rows at a time so
// that each lane keeps several loads in flight.  No shared memory, no barriers, no
// waits: nothing here can hang.
#include <cstdint>

#include "kvl_internal.cuh"

namespace kvl {
namespace {

enum Op { OP_SLICE = 0, OP_MERGE = 1, OP_GATHER = 2, OP_SCATTER = 3 };

constexpr int kThreads = 256;
constexpr int kMinBlocksPerSm = 4;
constexpr int kUnroll = 4;  // 16-byte vectors per lane per row per pass

struct CopyArgs {
    void *plan;
    const kvl_request *reqs;
    const int32_t *tables;
    uint8_t *pool;
    uint8_t *out;  // hit_out (slice), complete_out (merge, may be null)
    int32_t P, B, Rp, layer;
    int64_t N;
};

struct RowAddr {
    const uint8_t *src;
    uint8_t *dst;
    uint8_t *dst2;
};

__device__ __forceinline__ uint4 ld_stream(const uint8_t *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_global(uint8_t *p, const uint4 &v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// A plan is usable when it was built (magic) for this geometry, request array and
// block tables, and recorded no error.  The checks keep every later index inside
// the plan's own arrays and the request array it was sized for.
template <int OP>
__device__ __forceinline__ bool plan_usable(const CopyArgs &a)
{
    PlanHeader *h = static_cast<PlanHeader *>(a.plan);
    if (h->magic != kPlanMagic || h->pool_blocks != a.N || h->block_tokens != a.B ||
        h->reqs != a.reqs || (OP != OP_SLICE && h->tables != a.tables)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(h, KVL_EINVAL, 0);
        return false;
    }
    return h->status == KVL_OK;
}

// Addresses of row `row` of the op's row space (src == nullptr: nothing to copy).
template <int OP>
__device__ __forceinline__ RowAddr row_addr(const CopyArgs &a, const PlanView &v, int64_t row,
                                            int lane)
{
    RowAddr x{nullptr, nullptr, nullptr};
    const int rpi = OP == OP_SLICE ? a.B : a.P * a.B;
    const int64_t item = row / rpi;
    const int rem = int(row - item * rpi);
    const int p = OP == OP_SLICE ? 0 : rem / a.B;
    const int s = OP == OP_SLICE ? rem : rem - p * a.B;
    const int r = v.item_req[item];
    const int64_t j = v.item_blk[item];
    const kvl_request &q = a.reqs[r];
    const int64_t t = j * a.B + s;
    const int64_t Rp = a.Rp, R = int64_t(a.P) * a.Rp, l = a.layer;

    if (OP == OP_SLICE || OP == OP_MERGE) {
        const int64_t t_hit = q.t_hit, t_all = t_hit + q.t_miss;
        if (t >= (OP == OP_SLICE ? t_hit : t_all)) return x;
        const uint8_t *src;
        if (t < t_hit) {
            const int64_t sb = q.hit_src_table ? int64_t(q.hit_src_table[j]) : j;
            if (sb < 0 || sb >= q.hit_src_blocks) {
                if (lane == 0) record_error(v.hdr, KVL_ERANGE, (unsigned long long)item);
                return x;
            }
            src = static_cast<const uint8_t *>(q.hit_src) + sb * q.hit_block_stride +
                  s * q.hit_token_stride + l * q.hit_layer_stride + p * Rp;
        } else {
            src = static_cast<const uint8_t *>(q.miss_src) + (t - t_hit) * q.miss_token_stride +
                  l * q.miss_layer_stride + p * Rp;
        }
        if (OP == OP_SLICE) {
            x.src = src;
            x.dst = a.out + (v.hit_off[r] + t) * R;
            return x;
        }
        const int64_t b = a.tables[v.blk_off[r] + j];
        if (b < 0 || b >= a.N) {
            if (lane == 0) record_error(v.hdr, KVL_ERANGE, (unsigned long long)item);
            return x;
        }
        x.src = src;
        x.dst = a.pool + (((l * a.P + p) * a.N + b) * a.B + s) * Rp;
        if (a.out) x.dst2 = a.out + (v.tok_off[r] + t) * R + p * Rp;
        return x;
    } else {
        const int64_t b = a.tables[v.blk_off[r] + j];
        if (b < 0 || b >= a.N) {
            if (lane == 0) record_error(v.hdr, KVL_ERANGE, (unsigned long long)item);
            return x;
        }
        if (q.objects == nullptr) {
            if (lane == 0) record_error(v.hdr, KVL_EINVAL, (unsigned long long)r);
            return x;
        }
        const int64_t nblk = v.blk_off[r + 1] - v.blk_off[r];
        uint8_t *pool_row = a.pool + (((l * a.P + p) * a.N + b) * a.B + s) * Rp;
        uint8_t *obj_row = static_cast<uint8_t *>(q.objects) + l * q.obj_layer_stride +
                           ((p * nblk + j) * a.B + s) * Rp;
        if (OP == OP_GATHER) {
            x.src = pool_row;
            x.dst = obj_row;
        } else {
            x.src = obj_row;
            x.dst = pool_row;
        }
        return x;
    }
}

// Copy two rows of nvec 16-byte vectors; all loads of a pass are issued before its
// stores.
__device__ __forceinline__ void copy_pair(const RowAddr &a, const RowAddr &b, int nvec, int lane)
{
    for (int v0 = 0; v0 < nvec; v0 += 32 * kUnroll) {
        uint4 ra[kUnroll], rb[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int o = (v0 + k * 32 + lane) * 16;
            if (a.src && o < nvec * 16) ra[k] = ld_stream(a.src + o);
            if (b.src && o < nvec * 16) rb[k] = ld_stream(b.src + o);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int o = (v0 + k * 32 + lane) * 16;
            if (o < nvec * 16) {
                if (a.src) {
                    st_global(a.dst + o, ra[k]);
                    if (a.dst2) st_global(a.dst2 + o, ra[k]);
                }
                if (b.src) {
                    st_global(b.dst + o, rb[k]);
                    if (b.dst2) st_global(b.dst2 + o, rb[k]);
                }
            }
        }
    }
}

template <int OP>
__device__ __forceinline__ void copy_rows(const CopyArgs &a)
{
    if (!plan_usable<OP>(a)) return;
    const PlanHeader *h = static_cast<const PlanHeader *>(a.plan);
    const PlanView v = plan_view(a.plan, h->n_req, h->pool_blocks);
    const int rpi = OP == OP_SLICE ? a.B : a.P * a.B;
    const int nvec = (OP == OP_SLICE ? a.P * a.Rp : a.Rp) >> 4;
    const int64_t total = h->n_items * rpi;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (kThreads / 32);
    const int64_t w = int64_t(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    const int64_t begin = total * w / nwarps, end = total * (w + 1) / nwarps;
    for (int64_t row = begin; row < end; row += 2) {
        const RowAddr r0 = row_addr<OP>(a, v, row, lane);
        const RowAddr r1 = row + 1 < end ? row_addr<OP>(a, v, row + 1, lane) : RowAddr{nullptr, nullptr, nullptr};
        copy_pair(r0, r1, nvec, lane);
    }
}

// One kernel per op, so launch lists and profiles name the op.
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSm) kvl_slice_kernel(CopyArgs a)
{
    copy_rows<OP_SLICE>(a);
}
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSm) kvl_merge_scatter_kernel(CopyArgs a)
{
    copy_rows<OP_MERGE>(a);
}
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSm) kvl_gather_kernel(CopyArgs a)
{
    copy_rows<OP_GATHER>(a);
}
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSm) kvl_scatter_back_kernel(CopyArgs a)
{
    copy_rows<OP_SCATTER>(a);
}

template <int OP>
constexpr void (*kernel_of())(CopyArgs)
{
    return OP == OP_SLICE ? kvl_slice_kernel
         : OP == OP_MERGE ? kvl_merge_scatter_kernel
         : OP == OP_GATHER ? kvl_gather_kernel
                           : kvl_scatter_back_kernel;
}

template <int OP>
int grid_size()
{
    static int per_sm[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (per_sm[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel_of<OP>(), kThreads, 0) !=
                cudaSuccess ||
            n <= 0)
            return 0;
        per_sm[dev] = n;
    }
    return per_sm[dev] * sm_count();
}

template <int OP>
kvl_status launch(const CopyArgs &a, void *stream)
{
    const int grid = grid_size<OP>();
    if (grid <= 0) return KVL_ECUDA;
    kernel_of<OP>()<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return launch_status();
}

kvl_status common_checks(const kvl_geom *g, const void *d_plan, const kvl_request *d_reqs,
                         int32_t layer)
{
    const kvl_status s = check_geom(g);
    if (s) return s;
    if (!d_plan || !d_reqs) return KVL_EINVAL;
    if (!aligned16(d_plan) || !aligned16(d_reqs)) return KVL_EALIGN;
    if (layer < 0 || layer >= g->n_layers) return KVL_EINVAL;
    return KVL_OK;
}

CopyArgs make_args(const kvl_geom *g, const void *d_plan, const kvl_request *d_reqs,
                   const int32_t *tables, int32_t layer, void *pool, void *out)
{
    CopyArgs a;
    a.plan = const_cast<void *>(d_plan);
    a.reqs = d_reqs;
    a.tables = tables;
    a.pool = static_cast<uint8_t *>(pool);
    a.out = static_cast<uint8_t *>(out);
    a.P = g->n_planes;
    a.B = g->block_tokens;
    a.Rp = g->plane_row_bytes;
    a.layer = layer;
    a.N = g->pool_blocks;
    return a;
}

}  // namespace
}  // namespace kvl

using namespace kvl;

extern "C" kvl_status kvl_slice_layer(const kvl_geom *geom, const void *d_plan,
                                      const kvl_request *d_reqs, int32_t layer, void *d_hit_out,
                                      void *stream)
{
    kvl_status s = common_checks(geom, d_plan, d_reqs, layer);
    if (s) return s;
    if (!d_hit_out) return KVL_EINVAL;
    if (!aligned16(d_hit_out)) return KVL_EALIGN;
    return launch<OP_SLICE>(make_args(geom, d_plan, d_reqs, nullptr, layer, nullptr, d_hit_out),
                            stream);
}

extern "C" kvl_status kvl_merge_scatter_paged(const kvl_geom *geom, const void *d_plan,
                                              const kvl_request *d_reqs,
                                              const int32_t *d_block_tables, int32_t layer,
                                              void *d_pool, void *d_complete_out, void *stream)
{
    kvl_status s = common_checks(geom, d_plan, d_reqs, layer);
    if (s) return s;
    if (!d_block_tables || !d_pool) return KVL_EINVAL;
    if ((reinterpret_cast<uintptr_t>(d_block_tables) & 3u) || !aligned16(d_pool) ||
        (d_complete_out && !aligned16(d_complete_out)))
        return KVL_EALIGN;
    return launch<OP_MERGE>(
        make_args(geom, d_plan, d_reqs, d_block_tables, layer, d_pool, d_complete_out), stream);
}

extern "C" kvl_status kvl_gather_layer_objects(const kvl_geom *geom, const void *d_plan,
                                               const kvl_request *d_reqs,
                                               const int32_t *d_block_tables, int32_t layer,
                                               void *d_pool, int32_t direction, void *stream)
{
    kvl_status s = common_checks(geom, d_plan, d_reqs, layer);
    if (s) return s;
    if (!d_block_tables || !d_pool) return KVL_EINVAL;
    if (direction != KVL_GATHER && direction != KVL_SCATTER_BACK) return KVL_EINVAL;
    if ((reinterpret_cast<uintptr_t>(d_block_tables) & 3u) || !aligned16(d_pool)) return KVL_EALIGN;
    const CopyArgs a = make_args(geom, d_plan, d_reqs, d_block_tables, layer, d_pool, nullptr);
    return direction == KVL_GATHER ? launch<OP_GATHER>(a, stream) : launch<OP_SCATTER>(a, stream);
}

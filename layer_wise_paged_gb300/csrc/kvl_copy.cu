// kvl_copy.cu -- the per-layer copy kernels of libkvl.so: slice, merge-scatter into
// the paged pool, and gather / scatter-back of per-layer K/V objects.
//
// Every op walks a flat "row space": the rows of all work items of the plan, item by
// item (then plane by plane, then slot by slot).  A row is one token's Rp-byte plane
// (merge-scatter, gather, scatter-back) or one token's R-byte layer row (slice).
// Each CTA of a persistent grid takes one contiguous, equal share of the row space
// (balanced to within one row whatever the request mix) and cuts it into segments:
// runs of rows of one (item, plane) whose destination is one contiguous range, at
// most one shared-memory stage long.
//
// A CTA is one warp driving the Tensor Memory Accelerator's bulk copies:
//   * metadata: each lane decodes one work item (request, block, pool block id,
//     source block id, row bases) with plain loads, in parallel, and the warp reads
//     each item's fields from its owner lane with shuffles;
//   * loads: `cp.async.bulk` global -> shared, one per source row (rows of one token
//     plane are not adjacent in the full-block source), or one per segment when the
//     source run is contiguous (gather / scatter-back), completing on a stage's
//     mbarrier;
//   * stores: one `cp.async.bulk` shared -> global per segment (the destination run
//     is contiguous), in bulk groups; a stage is refilled only after its store has
//     read it (`cp.async.bulk.wait_group.read`).
// Loads run up to kStages - 1 segments ahead of stores, so each SM keeps well over
// 100 KiB in flight with no registers holding data.  Every mbarrier wait is bounded
// by the global timer: past the limit the kernel records KVL_ETIMEOUT, waits
// (bounded again) for its copies in flight and returns.
#include <cstdint>

#include "kvl_internal.cuh"

namespace kvl {
namespace {

enum Op { OP_SLICE = 0, OP_MERGE = 1, OP_GATHER = 2, OP_SCATTER = 3 };

#ifndef KVL_STAGES
#define KVL_STAGES 6
#endif
#ifndef KVL_STAGE_BYTES
#define KVL_STAGE_BYTES (32 * 1024)
#endif
#ifndef KVL_CTAS_PER_SM
#define KVL_CTAS_PER_SM 1
#endif
#ifndef KVL_PDL
#define KVL_PDL 1
#endif

constexpr int kStages = KVL_STAGES;
constexpr int kStageBytes = KVL_STAGE_BYTES;
constexpr int kCtasPerSm = KVL_CTAS_PER_SM;
constexpr int kLookahead = kStages - 1;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per mbarrier wait
static_assert(kStageBytes % 16 == 0 && kStages >= 2, "stage geometry");

struct CopyArgs {
    void *plan;
    const kvl_request *reqs;
    const int32_t *tables;
    uint8_t *pool;
    uint8_t *out;  // hit_out (slice), complete_out (merge, may be null)
    int32_t P, B, Rp, layer;
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
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
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

template <typename T>
__device__ __forceinline__ T shfl_ptr(T p, int src)
{
    return reinterpret_cast<T>(__shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(p), src));
}

// ---- plan checks and metadata ------------------------------------------------

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

// Decode work item `item` of layer a.layer.  Returns false (after recording the
// error) when a block id is out of range or a needed pointer is missing.
template <int OP>
__device__ bool item_meta(const CopyArgs &a, const PlanView &v, int64_t item, ItemMeta &m)
{
    const int r = v.item_req[item];
    const int64_t j = v.item_blk[item];
    const kvl_request &q = a.reqs[r];
    const int64_t B = a.B, Rp = a.Rp, l = a.layer, t0 = j * B;
    const int64_t t_hit = q.t_hit, t_all = t_hit + q.t_miss;
    m.src_a = m.src_b = nullptr;
    m.dst = m.dst2 = nullptr;
    m.a_stride = m.b_stride = m.src_pstride = m.dst_pstride = 0;
    const int64_t n_a = t_hit - t0 < 0 ? 0 : (t_hit - t0 > B ? B : t_hit - t0);
    const int64_t n_v = t_all - t0 < 0 ? 0 : (t_all - t0 > B ? B : t_all - t0);
    m.n_a = int32_t(n_a);
    m.n_valid = int32_t(n_v);

    if (OP == OP_SLICE || OP == OP_MERGE) {
        if (n_a > 0) {
            const int64_t sb = q.hit_src_table ? int64_t(q.hit_src_table[j]) : j;
            if (sb < 0 || sb >= q.hit_src_blocks) {
                record_error(v.hdr, KVL_ERANGE, (unsigned long long)item);
                return false;
            }
            m.src_a = static_cast<const uint8_t *>(q.hit_src) + sb * q.hit_block_stride +
                      l * q.hit_layer_stride;
            m.a_stride = q.hit_token_stride;
        }
        if (OP == OP_SLICE) {
            m.n_valid = m.n_a;
            m.dst = a.out + (v.hit_off[r] + t0) * (int64_t(a.P) * Rp);
            return true;
        }
        if (n_v > n_a) {
            // row s >= n_a is miss token t0 + s - t_hit
            m.src_b = static_cast<const uint8_t *>(q.miss_src) + (t0 - t_hit) * q.miss_token_stride +
                      l * q.miss_layer_stride;
            m.b_stride = q.miss_token_stride;
        }
        m.src_pstride = Rp;
        if (a.out) m.dst2 = a.out + (v.tok_off[r] + t0) * (int64_t(a.P) * Rp);
    }
    const int64_t b = a.tables[v.blk_off[r] + j];
    if (b < 0 || b >= a.N) {
        record_error(v.hdr, KVL_ERANGE, (unsigned long long)item);
        return false;
    }
    uint8_t *pool_blk = a.pool + ((l * a.P) * a.N + b) * B * Rp;
    const int64_t pool_pstride = a.N * B * Rp;
    if (OP == OP_MERGE) {
        m.dst = pool_blk;
        m.dst_pstride = pool_pstride;
        return true;
    }
    if (q.objects == nullptr) {
        record_error(v.hdr, KVL_EINVAL, (unsigned long long)r);
        return false;
    }
    const int64_t nblk = v.blk_off[r + 1] - v.blk_off[r];
    uint8_t *obj = static_cast<uint8_t *>(q.objects) + l * q.obj_layer_stride + j * B * Rp;
    const int64_t obj_pstride = nblk * B * Rp;
    m.n_a = m.n_valid = int32_t(B);  // objects carry whole blocks
    if (OP == OP_GATHER) {
        m.src_a = pool_blk;
        m.src_pstride = pool_pstride;
        m.dst = obj;
        m.dst_pstride = obj_pstride;
    } else {
        m.src_a = obj;
        m.src_pstride = obj_pstride;
        m.dst = pool_blk;
        m.dst_pstride = pool_pstride;
    }
    m.a_stride = Rp;
    return true;
}

__device__ __forceinline__ ItemMeta shfl_meta(const ItemMeta &m, int src)
{
    ItemMeta o;
    o.src_a = shfl_ptr(m.src_a, src);
    o.src_b = shfl_ptr(m.src_b, src);
    o.dst = shfl_ptr(m.dst, src);
    o.dst2 = shfl_ptr(m.dst2, src);
    o.a_stride = __shfl_sync(0xffffffffu, m.a_stride, src);
    o.b_stride = __shfl_sync(0xffffffffu, m.b_stride, src);
    o.src_pstride = __shfl_sync(0xffffffffu, m.src_pstride, src);
    o.dst_pstride = __shfl_sync(0xffffffffu, m.dst_pstride, src);
    o.n_a = __shfl_sync(0xffffffffu, m.n_a, src);
    o.n_valid = __shfl_sync(0xffffffffu, m.n_valid, src);
    return o;
}

// ---- the pipelined copy --------------------------------------------------------

struct StageInfo {
    uint8_t *dst;       // contiguous destination of the segment
    uint8_t *dst2;      // complete_layer row of the segment's first slot (or null)
    uint32_t bytes;     // segment bytes (= rows * row_bytes)
    uint32_t rows;
};

template <int OP>
__device__ __forceinline__ void copy_rows(const CopyArgs &a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kStages];
    __shared__ StageInfo info[kStages];

    const int lane = threadIdx.x;
    // Everything this kernel reads may come from the previous kernel on the stream.
    grid_dependency_wait();
    allow_dependents_launch();
    if (!plan_usable<OP>(a)) return;
    PlanHeader *h = static_cast<PlanHeader *>(a.plan);
    const PlanView v = plan_view(a.plan, h->n_req, h->pool_blocks);
    const int planes = OP == OP_SLICE ? 1 : a.P;
    const int rpi = planes * a.B;                        // rows per item
    const int row_bytes = OP == OP_SLICE ? a.P * a.Rp : a.Rp;
    const int max_rows = kStageBytes / row_bytes;        // >= 1 (host-checked)
    const int64_t total = h->n_items * rpi;
    const int64_t begin = total * blockIdx.x / gridDim.x;
    const int64_t end = total * (blockIdx.x + 1) / gridDim.x;
    if (begin >= end) return;
    const int64_t R = int64_t(a.P) * a.Rp;

    const uint32_t smem0 = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    int64_t issued = 0, retired = 0;
    bool timed_out = false;

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
        if (OP == OP_MERGE && si.dst2 != nullptr) {
            for (uint32_t i = lane; i < si.rows; i += 32)
                bulk_store(si.dst2 + int64_t(i) * R, src + i * uint32_t(row_bytes), uint32_t(row_bytes));
        }
        if (lane == 0) bulk_store(si.dst, src, si.bytes);
        bulk_commit();
        ++retired;
    };

    const int64_t item_first = begin / rpi;
    const int64_t item_last = (end - 1) / rpi;
    for (int64_t ib = item_first; ib <= item_last && !timed_out; ib += 32) {
        // each lane decodes one item of this batch
        ItemMeta mine{};
        bool ok_mine = false;
        if (ib + lane <= item_last) ok_mine = item_meta<OP>(a, v, ib + lane, mine);
        const unsigned ok_mask = __ballot_sync(0xffffffffu, ok_mine);
        const int nb = int(item_last - ib + 1 < 32 ? item_last - ib + 1 : 32);
        for (int k = 0; k < nb && !timed_out; ++k) {
            if (!((ok_mask >> k) & 1u)) continue;
            const ItemMeta m = shfl_meta(mine, k);
            const int64_t item = ib + k;
            const int64_t item_row0 = item * rpi;
            const int64_t lo = begin > item_row0 ? begin - item_row0 : 0;
            const int64_t hi = end - item_row0 < rpi ? end - item_row0 : rpi;
            for (int p = int(lo / a.B); p < planes && int64_t(p) * a.B < hi && !timed_out; ++p) {
                // slots [s_lo, s_hi) of plane p inside this CTA's share, clipped to valid rows
                int64_t s_lo = lo - int64_t(p) * a.B;
                if (s_lo < 0) s_lo = 0;
                int64_t s_hi = hi - int64_t(p) * a.B;
                if (s_hi > a.B) s_hi = a.B;
                if (s_hi > m.n_valid) s_hi = m.n_valid;
                for (int64_t s0 = s_lo; s0 < s_hi && !timed_out; s0 += max_rows) {
                    const int ns = int(s_hi - s0 < max_rows ? s_hi - s0 : max_rows);
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
                        si.dst = m.dst + p * m.dst_pstride + s0 * int64_t(row_bytes);
                        si.dst2 = (OP == OP_MERGE && m.dst2) ? m.dst2 + s0 * R + int64_t(p) * a.Rp
                                                             : nullptr;
                        si.bytes = bytes;
                        si.rows = uint32_t(ns);
                        info[st] = si;
                        mbar_arrive_expect_tx(bar, bytes);
                    }
                    __syncwarp();
                    if (OP == OP_GATHER || OP == OP_SCATTER) {
                        if (lane == 0)
                            bulk_load(sbase, m.src_a + p * m.src_pstride + s0 * int64_t(row_bytes), bytes, bar);
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
                }
            }
        }
    }
    while (retired < issued && !timed_out) retire();

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
}

// One kernel per op, so launch lists and profiles name the op.
__global__ void __launch_bounds__(32) kvl_slice_kernel(CopyArgs a) { copy_rows<OP_SLICE>(a); }
__global__ void __launch_bounds__(32) kvl_merge_scatter_kernel(CopyArgs a) { copy_rows<OP_MERGE>(a); }
__global__ void __launch_bounds__(32) kvl_gather_kernel(CopyArgs a) { copy_rows<OP_GATHER>(a); }
__global__ void __launch_bounds__(32) kvl_scatter_back_kernel(CopyArgs a) { copy_rows<OP_SCATTER>(a); }

template <int OP>
constexpr void (*kernel_of())(CopyArgs)
{
    return OP == OP_SLICE ? kvl_slice_kernel
         : OP == OP_MERGE ? kvl_merge_scatter_kernel
         : OP == OP_GATHER ? kvl_gather_kernel
                           : kvl_scatter_back_kernel;
}

constexpr int kSmemBytes = kStages * kStageBytes;

// Grid: kCtasPerSm CTAs on every SM; opts each kernel into its shared memory once
// per device.
template <int OP>
int grid_size()
{
    static bool ready[kMaxDevices] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (!ready[dev]) {
        if (cudaFuncSetAttribute(kernel_of<OP>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess)
            return 0;
        ready[dev] = true;
    }
    return kCtasPerSm * sm_count();
}

template <int OP>
kvl_status launch(const CopyArgs &a, void *stream)
{
    const int grid = grid_size<OP>();
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
    if (cudaLaunchKernelEx(&cfg, kernel_of<OP>(), a) != cudaSuccess) return KVL_ECUDA;
    return KVL_OK;
#else
    kernel_of<OP>()<<<grid, 32, kSmemBytes, static_cast<cudaStream_t>(stream)>>>(a);
    return launch_status();
#endif
}

kvl_status common_checks(const kvl_geom *g, const void *d_plan, const kvl_request *d_reqs,
                         int32_t layer, int32_t row_bytes)
{
    const kvl_status s = check_geom(g);
    if (s) return s;
    if (!d_plan || !d_reqs) return KVL_EINVAL;
    if (!aligned16(d_plan) || !aligned16(d_reqs)) return KVL_EALIGN;
    if (layer < 0 || layer >= g->n_layers) return KVL_EINVAL;
    if (row_bytes > kStageBytes) return KVL_EINVAL;  // a row must fit one stage
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
    const int32_t rb = geom ? geom->n_planes * geom->plane_row_bytes : 0;
    kvl_status s = common_checks(geom, d_plan, d_reqs, layer, rb);
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
    kvl_status s = common_checks(geom, d_plan, d_reqs, layer, geom ? geom->plane_row_bytes : 0);
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
    kvl_status s = common_checks(geom, d_plan, d_reqs, layer, geom ? geom->plane_row_bytes : 0);
    if (s) return s;
    if (!d_block_tables || !d_pool) return KVL_EINVAL;
    if (direction != KVL_GATHER && direction != KVL_SCATTER_BACK) return KVL_EINVAL;
    if ((reinterpret_cast<uintptr_t>(d_block_tables) & 3u) || !aligned16(d_pool)) return KVL_EALIGN;
    const CopyArgs a = make_args(geom, d_plan, d_reqs, d_block_tables, layer, d_pool, nullptr);
    return direction == KVL_GATHER ? launch<OP_GATHER>(a, stream) : launch<OP_SCATTER>(a, stream);
}

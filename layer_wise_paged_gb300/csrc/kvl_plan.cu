// kvl_plan.cu -- the batch plan (device-side prefix sums and work list), the status
// read-back, and the small host entry points of libkvl.so.
//
// The plan turns a batch of requests with ragged T_hit / T_miss into one flat list
// of (request, logical block) work items, so that each later per-layer call is a
// single launch over the whole batch (Tutti 阅读笔记, 伪代码 1 retrieve_layer: the
// CPU loads the I/O kernel once per layer, O(L) rather than O(L x blocks)).
//
// Two launches: a one-CTA scan (request validation, three exclusive prefix sums,
// header, claim counters and bitmap clear) and a grid-stride fill (work items,
// block-id range checks, optional injectivity check through a bitmap with atomicOr,
// and each item's resolved record: the layer-0 addresses and strides its rows are
// read from and written to, so the copy kernels need one 128-byte load per item).
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kvl_internal.cuh"

namespace kvl {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kFillThreads = 256;

struct PlanArgs {
    PlanView v;
    const kvl_request *reqs;
    const int32_t *tables;
    int32_t n_req;
    int32_t B;
    int64_t N;
    int32_t check_injective;
    int32_t P, Rp, L;
};

// Inclusive scan of one int64 across a warp.
__device__ __forceinline__ int64_t warp_inclusive(int64_t x, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    return x;
}

// Validate one request; returns the KVL code (0 = fine).
__device__ int validate_request(const kvl_request &q)
{
    if (q.t_hit < 0 || q.t_miss < 0) return KVL_EINVAL;
    if (q.t_hit > 0 && q.hit_src == nullptr) return KVL_EINVAL;
    if (q.t_miss > 0 && q.miss_src == nullptr) return KVL_EINVAL;
    if (q.t_hit > 0) {
        if (!aligned16(q.hit_src) || (q.hit_block_stride | q.hit_token_stride | q.hit_layer_stride) & 15)
            return KVL_EALIGN;
        if (q.hit_src_table && (reinterpret_cast<uintptr_t>(q.hit_src_table) & 3u)) return KVL_EALIGN;
    }
    if (q.t_miss > 0 && (!aligned16(q.miss_src) || (q.miss_token_stride | q.miss_layer_stride) & 15))
        return KVL_EALIGN;
    if (q.objects &&
        (!aligned16(q.objects) || ((q.obj_layer_stride | q.obj_plane_stride | q.obj_block_stride) & 15)))
        return KVL_EALIGN;
    return KVL_OK;
}

__global__ void __launch_bounds__(kScanThreads) plan_scan_kernel(PlanArgs a)
{
    __shared__ int64_t s_warp[3][kScanThreads / 32];
    __shared__ int64_t s_carry[3];
    __shared__ int s_code;
    __shared__ unsigned long long s_detail[8];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    PlanHeader *h = a.v.hdr;
    if (tid == 0) {
        s_code = KVL_OK;
        s_carry[0] = s_carry[1] = s_carry[2] = 0;
    }
    if (tid < 8) s_detail[tid] = ULLONG_MAX;
    __syncthreads();

    for (int base = 0; base < a.n_req; base += kScanThreads) {
        const int r = base + tid;
        int64_t ta = 0, th = 0, nb = 0;
        if (r < a.n_req) {
            const kvl_request q = a.reqs[r];
            const int code = validate_request(q);
            if (code) {
                atomicMax(&s_code, code);
                atomicMin(&s_detail[code], (unsigned long long)r);
            }
            th = q.t_hit > 0 ? q.t_hit : 0;
            ta = th + (q.t_miss > 0 ? q.t_miss : 0);
            nb = ceil_div64(ta, a.B);
        }
        const int64_t i0 = warp_inclusive(ta, lane);
        const int64_t i1 = warp_inclusive(th, lane);
        const int64_t i2 = warp_inclusive(nb, lane);
        if (lane == 31) {
            s_warp[0][warp] = i0;
            s_warp[1][warp] = i1;
            s_warp[2][warp] = i2;
        }
        __syncthreads();
        if (warp == 0) {
            for (int k = 0; k < 3; ++k) {
                const int64_t w = warp_inclusive(s_warp[k][lane], lane);
                s_warp[k][lane] = w;  // inclusive over warps
            }
        }
        __syncthreads();
        const int64_t w0 = warp ? s_warp[0][warp - 1] : 0;
        const int64_t w1 = warp ? s_warp[1][warp - 1] : 0;
        const int64_t w2 = warp ? s_warp[2][warp - 1] : 0;
        if (r < a.n_req) {
            a.v.tok_off[r] = s_carry[0] + w0 + i0 - ta;
            a.v.hit_off[r] = s_carry[1] + w1 + i1 - th;
            a.v.blk_off[r] = s_carry[2] + w2 + i2 - nb;
        }
        __syncthreads();
        if (tid == 0) {
            s_carry[0] += s_warp[0][31];
            s_carry[1] += s_warp[1][31];
            s_carry[2] += s_warp[2][31];
        }
        __syncthreads();
    }

    if (tid == 0) {
        a.v.tok_off[a.n_req] = s_carry[0];
        a.v.hit_off[a.n_req] = s_carry[1];
        a.v.blk_off[a.n_req] = s_carry[2];
        h->n_req = a.n_req;
        h->check_injective = a.check_injective;
        h->n_items = s_carry[2];
        h->n_tokens = s_carry[0];
        h->n_hit = s_carry[1];
        h->pool_blocks = a.N;
        h->block_tokens = a.B;
        int code = s_code;
        for (int k = 0; k < 8; ++k) h->detail[k] = s_detail[k];
        if (code == KVL_OK && s_carry[2] > a.N) {
            code = KVL_ERANGE;
            h->detail[KVL_ERANGE] = (unsigned long long)s_carry[2];
        }
        h->status = code;
        h->scan_status = code;
        h->n_layers = a.L;
        h->reqs = a.reqs;
        h->tables = a.tables;
        h->magic = kPlanMagic;
    }
    for (int64_t c = tid; c < int64_t(a.L) * kOps; c += kScanThreads) {
        a.v.counters[c].next = 0u;
        a.v.counters[c].done = 0u;
    }
    if (a.check_injective) {
        const int64_t words = (a.N + 31) / 32;
        for (int64_t w = tid; w < words; w += kScanThreads) a.v.bitmap[w] = 0u;
    }
}

__global__ void __launch_bounds__(kFillThreads) plan_fill_kernel(PlanArgs a)
{
    PlanHeader *h = a.v.hdr;
    // The scan's verdict, not `status`: other CTAs of this launch may already have
    // recorded errors there, and every item must still be checked.
    if (h->scan_status != KVL_OK) return;
    const int64_t n_items = h->n_items;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_items; i += stride) {
        // request r = the last one whose first item is <= i
        int lo = 0, hi = a.n_req;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (a.v.blk_off[mid] <= i) lo = mid; else hi = mid;
        }
        const int r = lo;
        const int64_t j = i - a.v.blk_off[r];
        a.v.item_req[i] = r;
        a.v.item_blk[i] = int32_t(j);

        const kvl_request &q = a.reqs[r];
        bool bad = false;
        int64_t sb = j;
        if (j < ceil_div64(q.t_hit, a.B)) {
            sb = q.hit_src_table ? int64_t(q.hit_src_table[j]) : j;
            if (sb < 0 || sb >= q.hit_src_blocks) bad = true;
        }
        const int64_t b = a.tables[i];
        if (b < 0 || b >= a.N) bad = true;
        if (bad) {
            record_error(h, KVL_ERANGE, (unsigned long long)i);
            continue;
        }
        if (a.check_injective) {
            const uint32_t bit = 1u << (b & 31);
            const uint32_t old = atomicOr(&a.v.bitmap[b >> 5], bit);
            if (old & bit) record_error(h, KVL_EDUP, (unsigned long long)b);
        }
        // the item's record
        const int64_t B = a.B, t0 = j * B;
        const int64_t t_hit = q.t_hit, t_all = t_hit + q.t_miss;
        const int64_t n_hit = t_hit - t0 < 0 ? 0 : (t_hit - t0 > B ? B : t_hit - t0);
        const int64_t n_valid = t_all - t0 < 0 ? 0 : (t_all - t0 > B ? B : t_all - t0);
        ItemRec rec;
        rec.hit_base = n_hit > 0 ? reinterpret_cast<uint64_t>(q.hit_src) + uint64_t(sb * q.hit_block_stride)
                                 : 0ull;
        rec.hit_ts = q.hit_token_stride;
        rec.hit_ls = q.hit_layer_stride;
        rec.miss_base = n_valid > n_hit ? reinterpret_cast<uint64_t>(q.miss_src) +
                                              uint64_t((t0 - t_hit) * q.miss_token_stride)
                                        : 0ull;
        rec.miss_ts = q.miss_token_stride;
        rec.miss_ls = q.miss_layer_stride;
        rec.obj_base = q.objects ? reinterpret_cast<uint64_t>(q.objects) + uint64_t(j * q.obj_block_stride)
                                 : 0ull;
        rec.obj_ps = q.obj_plane_stride;
        rec.obj_ls = q.obj_layer_stride;
        rec.hit_row = a.v.hit_off[r] + t0;
        rec.tok_row = a.v.tok_off[r] + t0;
        rec.pool_block = int32_t(b);
        rec.n_hit = int32_t(n_hit);
        rec.n_valid = int32_t(n_valid);
        rec.req = r;
        for (int k = 0; k < 6; ++k) rec.pad[k] = 0;
        a.v.items[i] = rec;
    }
}

}  // namespace
}  // namespace kvl

using namespace kvl;

extern "C" size_t kvl_plan_bytes(const kvl_geom *geom, int32_t n_req)
{
    if (check_geom(geom) != KVL_OK) return 0;
    return plan_layout(n_req, geom->pool_blocks, geom->n_layers).off[9];
}

extern "C" void kvl_plan_layout(const kvl_geom *geom, int32_t n_req, size_t off[10])
{
    if (!off) return;
    if (check_geom(geom) != KVL_OK) {
        for (int k = 0; k < 10; ++k) off[k] = 0;
        return;
    }
    const PlanLayout l = plan_layout(n_req, geom->pool_blocks, geom->n_layers);
    for (int k = 0; k < 10; ++k) off[k] = l.off[k];
}

extern "C" kvl_status kvl_batch_plan(const kvl_geom *geom, int32_t n_req, const kvl_request *d_reqs,
                                     const int32_t *d_block_tables, int32_t check_injective,
                                     void *d_plan, size_t plan_bytes, void *stream)
{
    const kvl_status g = check_geom(geom);
    if (g) return g;
    if (n_req < 0 || !d_plan) return KVL_EINVAL;
    if (n_req > 0 && (!d_reqs || !d_block_tables)) return KVL_EINVAL;
    if (!aligned16(d_plan) || (d_reqs && !aligned16(d_reqs)) ||
        (reinterpret_cast<uintptr_t>(d_block_tables) & 3u))
        return KVL_EALIGN;
    if (plan_bytes < kvl_plan_bytes(geom, n_req)) return KVL_EINVAL;

    PlanArgs a;
    a.v = plan_view(d_plan, n_req, geom->pool_blocks, geom->n_layers);
    a.reqs = d_reqs;
    a.tables = d_block_tables;
    a.n_req = n_req;
    a.B = geom->block_tokens;
    a.N = geom->pool_blocks;
    a.check_injective = check_injective ? 1 : 0;
    a.P = geom->n_planes;
    a.Rp = geom->plane_row_bytes;
    a.L = geom->n_layers;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    plan_scan_kernel<<<1, kScanThreads, 0, s>>>(a);
    if (launch_status()) return KVL_ECUDA;
    const int sms = sm_count();
    if (sms <= 0) return KVL_ECUDA;
    // Enough threads for one pass over the pool's worth of items on most batches.
    int64_t want = (geom->pool_blocks + kFillThreads - 1) / kFillThreads;
    int grid = int(want < int64_t(sms) * 4 ? (want < 1 ? 1 : want) : int64_t(sms) * 4);
    plan_fill_kernel<<<grid, kFillThreads, 0, s>>>(a);
    return launch_status();
}

extern "C" kvl_status kvl_read_status(const void *d_plan, int32_t *code, int64_t *detail, void *stream)
{
    if (!d_plan) return KVL_EINVAL;
    PlanHeader h;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&h, d_plan, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KVL_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVL_ECUDA;
    int32_t c = h.magic == kPlanMagic ? h.status : KVL_EINVAL;
    if (c < 0 || c > 7) c = KVL_EINVAL;
    if (code) *code = c;
    if (detail) *detail = (c == KVL_OK || h.magic != kPlanMagic) ? 0 : (int64_t)h.detail[c];
    return KVL_OK;
}

extern "C" const char *kvl_status_string(kvl_status s)
{
    switch (s) {
    case KVL_OK: return "ok";
    case KVL_EINVAL: return "invalid argument";
    case KVL_EALIGN: return "misaligned pointer, stride or row size (16 bytes required)";
    case KVL_ERANGE: return "block id out of range or plan capacity exceeded";
    case KVL_EDUP: return "pool block id used twice";
    case KVL_ECUDA: return "CUDA error";
    case KVL_ETIMEOUT: return "a copy kernel's bounded wait on its own copies ran out";
    default: return "unknown status";
    }
}

extern "C" int32_t kvl_launches_per_call(int32_t which)
{
    switch (which) {
    case 0: return 2;  // plan: scan + fill
    case 1: case 2: case 3: return 1;
    default: return 0;
    }
}

// ---------------------------------------------------------------------------
// kvl_batch_plan_static_scratch: the plan builder for callers that cannot
// allocate device memory.  Its only scratch, the injectivity bitmap, lives in the
// file-scope array below instead of the caller's plan buffer.  The array is a
// fixed KVL_STATIC_SCRATCH_POOL_BLOCKS / 8 bytes (512 KiB) that every GPU which
// loads this library holds until the process exits.
// ---------------------------------------------------------------------------

namespace kvl {
namespace {

static __device__ __align__(256) uint32_t g_plan_bitmap[KVL_STATIC_SCRATCH_POOL_BLOCKS / 32];

// Host code must not pass g_plan_bitmap itself to a kernel: on the host that name
// is a stand-in, not a device address.  The device address is looked up once per
// device, with that device current, and cached here.
uint32_t *g_plan_bitmap_dev[kMaxDevices] = {nullptr};
std::mutex g_plan_bitmap_mutex;

kvl_status static_bitmap_address(uint32_t **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVL_ECUDA;
    std::lock_guard<std::mutex> lock(g_plan_bitmap_mutex);
    if (g_plan_bitmap_dev[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_plan_bitmap) != cudaSuccess || p == nullptr) return KVL_ECUDA;
        g_plan_bitmap_dev[dev] = static_cast<uint32_t *>(p);
    }
    *out = g_plan_bitmap_dev[dev];
    return KVL_OK;
}

}  // namespace
}  // namespace kvl

extern "C" kvl_status kvl_batch_plan_static_scratch(const kvl_geom *geom, int32_t n_req,
                                                    const kvl_request *d_reqs,
                                                    const int32_t *d_block_tables,
                                                    int32_t check_injective, void *d_plan,
                                                    size_t plan_bytes, void *stream)
{
    const kvl_status g = check_geom(geom);
    if (g) return g;
    if (geom->pool_blocks > KVL_STATIC_SCRATCH_POOL_BLOCKS) return KVL_EINVAL;
    if (n_req < 0 || !d_plan) return KVL_EINVAL;
    if (n_req > 0 && (!d_reqs || !d_block_tables)) return KVL_EINVAL;
    if (!aligned16(d_plan) || (d_reqs && !aligned16(d_reqs)) ||
        (reinterpret_cast<uintptr_t>(d_block_tables) & 3u))
        return KVL_EALIGN;
    // everything of the plan but its bitmap section
    if (plan_bytes < plan_layout(n_req, geom->pool_blocks, geom->n_layers).off[8]) return KVL_EINVAL;

    uint32_t *bitmap = nullptr;
    const kvl_status sa = static_bitmap_address(&bitmap);
    if (sa) return sa;

    PlanArgs a;
    a.v = plan_view(d_plan, n_req, geom->pool_blocks, geom->n_layers);
    a.v.bitmap = bitmap;  // the scan kernel clears the words it uses on every call
    a.reqs = d_reqs;
    a.tables = d_block_tables;
    a.n_req = n_req;
    a.B = geom->block_tokens;
    a.N = geom->pool_blocks;
    a.check_injective = check_injective ? 1 : 0;
    a.P = geom->n_planes;
    a.Rp = geom->plane_row_bytes;
    a.L = geom->n_layers;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    plan_scan_kernel<<<1, kScanThreads, 0, s>>>(a);
    if (launch_status()) return KVL_ECUDA;
    const int sms = sm_count();
    if (sms <= 0) return KVL_ECUDA;
    int64_t want = (geom->pool_blocks + kFillThreads - 1) / kFillThreads;
    int grid = int(want < int64_t(sms) * 4 ? (want < 1 ? 1 : want) : int64_t(sms) * 4);
    plan_fill_kernel<<<grid, kFillThreads, 0, s>>>(a);
    return launch_status();
}

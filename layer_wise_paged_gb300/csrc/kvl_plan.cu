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

#include <cuda.h>
#include <cudaTypedefs.h>

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
    int32_t map_chunk;  // bytes per chunk of a map row; 0: build no tensor maps
    int32_t map_ops;    // map_bit(kind) for every map kind this geometry allows
    // Host-encoded maps that the fill kernel copies and edits, by row width (0: plane
    // rows, for the hit and miss maps; 1: token rows, for the slice maps), dim order
    // (0: token first; 1: layer first) and box height (0: a whole segment; 1: a block
    // tail).  Each already has its final box: the encoder derives more from the box
    // than the box dims themselves, so only the address, dims and strides are edited
    // on the device.
    CUtensorMap tmpl[2][2][2];
};

// Row width, box height and box rows of a map kind.
__host__ __device__ inline bool kind_token_rows(int kind) { return kind == MAP_SLICE || kind == MAP_SLICE_TAIL; }
__host__ __device__ inline bool kind_tail(int kind) { return kind >= kMapTail; }
__host__ __device__ inline int32_t kind_rows(int kind, int32_t B, int32_t P, int32_t Rp)
{
    const int32_t w = kind_token_rows(kind) ? P * Rp : Rp;
    return kind_tail(kind) ? segment_tail_rows(B, w) : segment_rows(B, w);
}

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

// ---- tensor maps ---------------------------------------------------------------

// The fields of one tensor map: a source's rows viewed as the 5-D tensor described
// with kMapBytes in kvl_internal.cuh.
struct MapShape {
    uint64_t base;
    uint32_t dim[5];
    uint64_t stride[4];  // bytes; stride[i] belongs to dim i + 1
    bool layer_first;    // dims 2, 3 are (layer, token) rather than (token, layer); the
                         // box (from the template) has its rows along the token dim
};

constexpr int64_t kMaxMapStride = int64_t(1) << 40;  // strides stay below 2^40 bytes
// The host encoder sets a flag in a map from the extent of memory the map spans (it
// differs below and above 128 KiB), which editing dims and strides on the device
// does not update.  So every template spans at least kTemplateSpan, and the plan
// builds maps only for views that span at least kMinMapSpan along one dim; smaller
// sources (a few hundred KiB at most) keep the per-row loads.
constexpr int64_t kMinMapSpan = int64_t(1) << 20;
constexpr int64_t kTemplateSpan = int64_t(1) << 21;

// Rows of R bytes at base + tok*ts + lay*ls + blk*bs, tok < n_tok, lay < L,
// blk < n_blk, read through boxes of `rows` token rows.  True, with the map's
// fields, when those rows are a non-overlapping strided view (each stride at least
// the extent below it) at least one box high; otherwise the per-row loads serve the
// source.
__device__ bool map_shape(uint64_t base, int64_t n_tok, int64_t ts, int64_t L, int64_t ls,
                          int64_t n_blk, int64_t bs, int32_t R, int32_t C, int32_t rows,
                          MapShape &m)
{
    if (base == 0 || n_tok < rows || L < 1 || n_blk < 1 || n_tok > INT32_MAX || L > INT32_MAX ||
        n_blk > INT32_MAX)
        return false;
    // the smaller stride first; a dim of extent one gets the stride that keeps the
    // view monotonic
    const bool layer_first = L > 1 && (n_tok == 1 || ls < ts);
    const int64_t e_in = layer_first ? L : n_tok, e_out = layer_first ? n_tok : L;
    int64_t s_in = layer_first ? ls : ts, s_out = layer_first ? ts : ls;
    if (e_in == 1) s_in = R;
    if (s_in < R || s_in >= kMaxMapStride) return false;
    if (e_out == 1) {
        if (s_in > kMaxMapStride / e_in) return false;
        s_out = e_in * s_in;
    } else if (s_out / e_in < s_in) {
        return false;
    }
    if (s_out >= kMaxMapStride) return false;
    if (n_blk == 1) {
        if (s_out > kMaxMapStride / e_out) return false;
        bs = e_out * s_out;
    } else if (bs / e_out < s_out) {
        return false;
    }
    if (bs >= kMaxMapStride) return false;
    // some dim's (extent - 1) x stride reaches kMinMapSpan (compared by division:
    // the block dim's product may exceed 64 bits)
    auto reaches = [](int64_t count, int64_t stride) {
        return count > 0 && stride > 0 && count >= (kMinMapSpan + stride - 1) / stride;
    };
    if (!(reaches(C / 8 - 1, 8) || reaches(R / C - 1, C) || reaches(e_in - 1, s_in) ||
          reaches(e_out - 1, s_out) || reaches(n_blk - 1, bs)))
        return false;
    m.base = base;
    m.layer_first = layer_first;
    m.dim[0] = uint32_t(C / 8);
    m.dim[1] = uint32_t(R / C);
    m.dim[2] = uint32_t(e_in);
    m.dim[3] = uint32_t(e_out);
    m.dim[4] = uint32_t(n_blk);
    m.stride[0] = uint64_t(C);
    m.stride[1] = uint64_t(s_in);
    m.stride[2] = uint64_t(s_out);
    m.stride[3] = uint64_t(bs);
    return true;
}

// The tensor maps request q gets (map_bit flags and the dim-order flags), and their
// fields if `shapes` is not null.  Hit rows: with a full-block table, blocks of B
// token rows (every one of the hit_src_blocks blocks is whole); without one, T_hit
// token rows when consecutive blocks follow one another (block stride = B x token
// stride, or a single block).  All maps of one source share its view, so its dim
// order.
__device__ int32_t request_maps(const PlanArgs &a, const kvl_request &q, MapShape *shapes)
{
    if (!a.map_ops) return 0;
    MapShape scratch;  // the flags alone need no shapes kept
    auto sh_of = [&](int k) -> MapShape & { return shapes ? shapes[k] : scratch; };
    const int32_t C = a.map_chunk, R = a.P * a.Rp;
    const int64_t B = a.B;
    int32_t flags = 0;
    if (q.t_hit > 0) {
        const uint64_t base = reinterpret_cast<uint64_t>(q.hit_src);
        const int64_t ts = q.hit_token_stride, bs = q.hit_block_stride;
        int64_t n_tok = 0, n_blk = 0;
        if (q.hit_src_table) {
            n_tok = B;
            n_blk = q.hit_src_blocks;
        } else if (q.t_hit <= B || (ts > 0 && bs % B == 0 && bs / B == ts)) {
            n_tok = q.t_hit;
            n_blk = 1;
        }
        const int hit_kinds[4] = {MAP_HIT, MAP_SLICE, MAP_HIT_TAIL, MAP_SLICE_TAIL};
        for (int i = 0; i < 4 && n_tok > 0; ++i) {
            const int k = hit_kinds[i];
            MapShape &sh = sh_of(k);
            if ((a.map_ops & map_bit(k)) &&
                map_shape(base, n_tok, ts, a.L, q.hit_layer_stride, n_blk, bs, R, C,
                          kind_rows(k, a.B, a.P, a.Rp), sh))
                flags |= map_bit(k) | (sh.layer_first ? kMapHitLayerFirst : 0);
        }
    }
    if (q.t_miss > 0) {
        const int miss_kinds[2] = {MAP_MISS, MAP_MISS_TAIL};
        for (int i = 0; i < 2; ++i) {
            const int k = miss_kinds[i];
            MapShape &sh = sh_of(k);
            if ((a.map_ops & map_bit(k)) &&
                map_shape(reinterpret_cast<uint64_t>(q.miss_src), q.t_miss, q.miss_token_stride,
                          a.L, q.miss_layer_stride, 1, 0, R, C, kind_rows(k, a.B, a.P, a.Rp), sh))
                flags |= map_bit(k) | (sh.layer_first ? kMapMissLayerFirst : 0);
        }
    }
    return flags;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Write the address, dims and strides of `m` into the map in shared memory at `s`
// (a copy of the template whose box m.box already is).
__device__ __forceinline__ void map_replace(uint32_t s, const MapShape &m)
{
    asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;" ::"r"(s),
                 "l"(m.base) : "memory");
#define KVL_MAP_DIM(i)                                                                              \
    asm volatile("tensormap.replace.tile.global_dim.shared::cta.b1024.b32 [%0], " #i ", %1;" ::"r"(s), \
                 "r"(m.dim[i]) : "memory");
#define KVL_MAP_STRIDE(i)                                                                           \
    asm volatile("tensormap.replace.tile.global_stride.shared::cta.b1024.b64 [%0], " #i ", %1;" ::"r"(s), \
                 "l"(m.stride[i]) : "memory");
    KVL_MAP_DIM(0) KVL_MAP_DIM(1) KVL_MAP_DIM(2) KVL_MAP_DIM(3) KVL_MAP_DIM(4)
    KVL_MAP_STRIDE(0) KVL_MAP_STRIDE(1) KVL_MAP_STRIDE(2) KVL_MAP_STRIDE(3)
#undef KVL_MAP_DIM
#undef KVL_MAP_STRIDE
}

// One warp per request: copy the template into shared memory, replace its fields,
// and copy it to the plan with a release to the tensor-map proxy (the copy kernels
// acquire each map before their first tensor load through it).
__device__ void build_maps(const PlanArgs &a)
{
    constexpr int kWarps = kFillThreads / 32;
    __shared__ __align__(128) uint8_t s_map[kWarps][kMapBytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t sm = smem_addr(s_map[warp]);
    const int64_t n_warps = int64_t(gridDim.x) * kWarps;
    for (int64_t r = int64_t(blockIdx.x) * kWarps + warp; r < a.n_req; r += n_warps) {
        const kvl_request q = a.reqs[r];
        MapShape sh[kMapsPerReq];
        const int32_t flags = request_maps(a, q, sh);  // = map_flags[r], with the shapes
        for (int k = 0; k < kMapsPerReq; ++k) {
            if (!(flags & map_bit(k))) continue;
            const uint4 *tmpl = reinterpret_cast<const uint4 *>(
                &a.tmpl[kind_token_rows(k) ? 1 : 0][sh[k].layer_first ? 1 : 0][kind_tail(k) ? 1 : 0]);
            if (lane < kMapBytes / 16) reinterpret_cast<uint4 *>(s_map[warp])[lane] = tmpl[lane];
            __syncwarp();
            if (lane == 0) map_replace(sm, sh[k]);
            __syncwarp();
            uint8_t *g = a.v.maps + (r * kMapsPerReq + k) * kMapBytes;
            asm volatile(
                "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned "
                "[%0], [%1], 128;" ::"l"(g),
                "r"(sm)
                : "memory");
            __syncwarp();
        }
    }
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
            // the request's tensor maps (the fill kernel builds them and stamps these
            // flags into the request's item records); none for an invalid request
            a.v.map_flags[r] = code ? 0 : request_maps(a, q, nullptr);
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
        h->map_chunk = a.map_ops ? a.map_chunk : 0;
        h->n_planes = a.P;
        h->plane_row_bytes = a.Rp;
        h->pad0 = 0;
        h->magic = kPlanMagic;
    }
    for (int64_t c = tid; c < int64_t(a.L) * kOps; c += kScanThreads) {
        a.v.counters[c].next = 0u;
        a.v.counters[c].reserved = 0u;
    }
    if (a.check_injective) {
        const int64_t words = (a.N + 31) / 32;
        for (int64_t w = tid; w < words; w += kScanThreads) a.v.bitmap[w] = 0u;
    }
}

__global__ void __launch_bounds__(kFillThreads) plan_fill_kernel(const __grid_constant__ PlanArgs a)
{
    PlanHeader *h = a.v.hdr;
    // The scan's verdict, not `status`: other CTAs of this launch may already have
    // recorded errors there, and every item must still be checked.
    if (h->scan_status != KVL_OK) return;
    if (a.map_ops) build_maps(a);
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
        rec.hit_blk_crd = q.hit_src_table ? int32_t(sb) : 0;
        rec.hit_tok_crd = q.hit_src_table ? 0 : int32_t(t0);
        rec.miss_tok_crd = int32_t(t0 - t_hit);
        rec.map_flags = a.v.map_flags[r];
        rec.pad[0] = rec.pad[1] = 0;
        a.v.items[i] = rec;
    }
}

// ---- host side ---------------------------------------------------------------

// cuTensorMapEncodeTiled, looked up once through the runtime (no link to the driver
// library); null if the driver does not offer it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A map a plan's tensor maps start from: rank 5, 8-byte elements, no interleave or
// swizzle, L2 promotion in 128-byte lines, zero fill out of bounds, and the box of
// `rows` token rows of W bytes (chunks of C bytes), the rows along dim 2 (token
// first) or dim 3 (layer first).  Its address, dims and strides are placeholders
// that the fill kernel replaces; it spans kTemplateSpan bytes along dim 4, as
// large a span class as every view the plan builds maps for.
bool encode_template(CUtensorMap *t, void *addr, int32_t C, int32_t R, int32_t W, int32_t rows,
                     bool layer_first)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t e = cuuint64_t(rows < 2 ? 2 : rows);
    const cuuint64_t dims[5] = {cuuint64_t(C / 8), cuuint64_t(R / C), e, e, 2};
    const cuuint64_t packed = cuuint64_t(R) * e * e;
    const cuuint64_t strides[4] = {cuuint64_t(C), cuuint64_t(R), cuuint64_t(R) * e,
                                   packed > cuuint64_t(kTemplateSpan) ? packed
                                                                      : cuuint64_t(kTemplateSpan)};
    const cuuint32_t box[5] = {cuuint32_t(C / 8), cuuint32_t(W / C),
                               layer_first ? 1u : cuuint32_t(rows), layer_first ? cuuint32_t(rows) : 1u,
                               1u};
    const cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    return enc(t, CU_TENSOR_MAP_DATA_TYPE_UINT64, 5, addr, dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The map kinds a geometry allows: a box is at most 256 elements along each dim, a
// slice row must fit one stage, and a tail kind exists only where blocks have a tail.
int32_t geometry_map_ops(const kvl_geom *g, int32_t C)
{
    if (C <= 0) return 0;
    const int64_t Rp = g->plane_row_bytes, R = int64_t(g->n_planes) * Rp;
    int32_t ops = 0;
    for (int k = 0; k < kMapsPerReq; ++k) {
        const int64_t w = kind_token_rows(k) ? R : Rp;
        if (w > kStageBytes || w / C > 256 || R / C > INT32_MAX) continue;
        const int32_t rows = kind_rows(k, g->block_tokens, g->n_planes, g->plane_row_bytes);
        if (rows >= 1 && rows <= 256) ops |= map_bit(k);
    }
    return ops;
}

// Arguments of the two plan kernels (the caller has checked geom and d_plan).
PlanArgs plan_args(const kvl_geom *geom, int32_t n_req, const kvl_request *d_reqs,
                   const int32_t *d_block_tables, int32_t check_injective, void *d_plan)
{
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
    a.map_chunk = map_chunk_bytes(geom->plane_row_bytes);
    a.map_ops = geometry_map_ops(geom, a.map_chunk);
    std::memset(&a.tmpl, 0, sizeof(a.tmpl));
    const int32_t C = a.map_chunk, R = a.P * a.Rp;
    // one template per (row width, dim order, box height); the kinds that share one
    // (hit and miss plane rows) share it
    for (int k = 0; k < kMapsPerReq; ++k) {
        if (!(a.map_ops & map_bit(k)) || k == MAP_MISS || k == MAP_MISS_TAIL) continue;
        const int width = kind_token_rows(k) ? 1 : 0, height = kind_tail(k) ? 1 : 0;
        const int32_t rows = kind_rows(k, a.B, a.P, a.Rp);
        for (int order = 0; order < 2; ++order) {
            if (encode_template(&a.tmpl[width][order][height], d_plan, C, R, width ? R : a.Rp,
                                rows, order != 0))
                continue;
            a.map_ops &= ~map_bit(k);  // and the miss kind that shares the template
            if (k == MAP_HIT) a.map_ops &= ~map_bit(MAP_MISS);
            if (k == MAP_HIT_TAIL) a.map_ops &= ~map_bit(MAP_MISS_TAIL);
        }
    }
    return a;
}

kvl_status launch_plan(const PlanArgs &a, int64_t pool_blocks, void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    plan_scan_kernel<<<1, kScanThreads, 0, s>>>(a);
    if (launch_status()) return KVL_ECUDA;
    const int sms = sm_count();
    if (sms <= 0) return KVL_ECUDA;
    // Enough threads for one pass over the pool's worth of items on most batches.
    int64_t want = (pool_blocks + kFillThreads - 1) / kFillThreads;
    int grid = int(want < int64_t(sms) * 4 ? (want < 1 ? 1 : want) : int64_t(sms) * 4);
    plan_fill_kernel<<<grid, kFillThreads, 0, s>>>(a);
    return launch_status();
}

}  // namespace
}  // namespace kvl

using namespace kvl;

extern "C" size_t kvl_plan_bytes(const kvl_geom *geom, int32_t n_req)
{
    if (check_geom(geom) != KVL_OK) return 0;
    return plan_layout(n_req, geom->pool_blocks, geom->n_layers).off[9];
}

extern "C" void kvl_plan_layout(const kvl_geom *geom, int32_t n_req, size_t off[11])
{
    if (!off) return;
    if (check_geom(geom) != KVL_OK) {
        for (int k = 0; k < 11; ++k) off[k] = 0;
        return;
    }
    const PlanLayout l = plan_layout(n_req, geom->pool_blocks, geom->n_layers);
    for (int k = 0; k < 11; ++k) off[k] = l.off[k];
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
    return launch_plan(plan_args(geom, n_req, d_reqs, d_block_tables, check_injective, d_plan),
                       geom->pool_blocks, stream);
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
// is a stand-in, not a device address.  The device address belongs to the module
// loaded into one CUDA context, and a new context (after cudaDeviceReset, or another
// context made current) loads the module again, possibly elsewhere.  So the address
// is looked up again, with the device current, on every call that is not being
// captured into a graph, and cached with the unique id of the context it belongs to;
// a call under capture uses the cache only when that id is the current context's, and
// otherwise refuses (a lookup is not a stream operation a graph could hold).
struct BitmapAddress {
    unsigned long long ctx_id = 0;
    uint32_t *ptr = nullptr;
};
BitmapAddress g_plan_bitmap_dev[kMaxDevices];
std::mutex g_plan_bitmap_mutex;

kvl_status static_bitmap_address(cudaStream_t stream, uint32_t **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVL_ECUDA;
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) return KVL_ECUDA;
    std::lock_guard<std::mutex> lock(g_plan_bitmap_mutex);
    BitmapAddress &c = g_plan_bitmap_dev[dev];
    if (capture == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_plan_bitmap) != cudaSuccess || p == nullptr) return KVL_ECUDA;
        c.ptr = static_cast<uint32_t *>(p);
        c.ctx_id = current_context_id();
    } else {
        const unsigned long long id = current_context_id();
        if (c.ptr == nullptr || id == 0 || id != c.ctx_id) return KVL_ECUDA;
    }
    *out = c.ptr;
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
    const kvl_status sa = static_bitmap_address(static_cast<cudaStream_t>(stream), &bitmap);
    if (sa) return sa;

    PlanArgs a = plan_args(geom, n_req, d_reqs, d_block_tables, check_injective, d_plan);
    a.v.bitmap = bitmap;  // the scan kernel clears the words it uses on every call
    return launch_plan(a, geom->pool_blocks, stream);
}

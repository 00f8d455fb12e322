/*
 * kvl.h -- layer-wise paged KV block reshuffle on one GPU (GB300, sm_103a).
 *
 * C ABI of libkvl.so.  Every buffer is caller memory; the library allocates nothing,
 * keeps no per-call state and never synchronises the caller's stream except in
 * kvl_read_status.  All calls only ENQUEUE work on `stream` (a cudaStream_t passed as
 * void*, NULL = the legacy default stream): results are valid once the caller has
 * synchronised that stream or an event recorded after the call (DualPath KV Loading,
 * "Dual-Path Loading", pe_read_path listing: every write is followed by a wait for
 * its completion before the buffer is used).
 *
 * What the calls compute (the pages' objects, per layer l):
 *   hit_full_block       persisted cross-layer KV of the hit prefix, semantic view
 *                        [T_hit, L, C_KV]; here [T_hit, L, P, Rp] bytes, token-major
 *                        (DualPath KV Loading, "Dual-Path Loading", objects table)
 *   hit_layer[l]         = hit_full_block[:, l], [T_hit, P, Rp]          (slice_layer)
 *   miss_layer[l]        freshly computed KV of the appended tokens, [T_miss, P, Rp]
 *   complete_layer[l]    hit rows then miss rows, [T_all, P, Rp]   (concatenate_tokens)
 *   paged pool           blocks of [B_tokens, H, d] linked per sequence by a block
 *                        table (Tutti 阅读笔记, 前置知识 3 "分页 KV 内存管理", eq. (2))
 *   K / V objects        one K and one V object per (layer, block): 2*L*ceil(T/B)
 *                        objects per sequence (Tutti 阅读笔记, 前置知识 5, eqs. (3)(4);
 *                        设计一 §3.1: one GPU file per block holding 2L objects)
 *
 * Geometry symbols: L layers, P planes per token (2 = K and V for head-split KV,
 * 1 = one latent vector), B tokens per block, Rp bytes per token per plane
 * (H_kv*d*2 for bf16 heads, C_KV*2 for a bf16 latent vector), R = P*Rp, N pool blocks.
 * T_all = T_hit + T_miss, nblk = ceil(T_all / B), nsrc = ceil(T_hit / B).
 *
 * Layouts (byte addresses; every one is a plain byte copy, values never pass through
 * arithmetic, so the results are bit-exact):
 *   hit token t (t < T_hit), layer l, plane p:
 *       hit_src + sb(t/B)*hit_block_stride + (t%B)*hit_token_stride
 *               + l*hit_layer_stride + p*Rp,   sb(j) = hit_src_table ? hit_src_table[j] : j
 *       (a contiguous full block [T_hit, L, P, Rp] has block stride B*L*R, token
 *        stride L*R, layer stride R; a "Full Block" store of [B, L, P, Rp] blocks at
 *        shuffled places uses hit_src_table)
 *   miss token t (T_hit <= t < T_all):
 *       miss_src + (t - T_hit)*miss_token_stride + l*miss_layer_stride + p*Rp
 *   pool, block b, slot s:  pool + (((l*P + p)*N + b)*B + s)*Rp   ([L][P][N][B][Rp])
 *   object (l, p, j) of a request, B*Rp bytes:
 *       objects + l*obj_layer_stride + p*obj_plane_stride + j*obj_block_stride
 *       layer-major [L][P][nblk][B][Rp] (object id (l*P + p)*nblk + j): strides
 *         (P*nblk*B*Rp, nblk*B*Rp, B*Rp);
 *       block-major [nblk][L][P][B][Rp], one "GPU file" per block holding its 2L
 *         objects (Tutti 阅读笔记, 设计一 §3.1 and 伪代码 1: file offset = file id x
 *         file stride + layer x per-layer size): strides (P*B*Rp, B*Rp, L*P*B*Rp)
 *   hit_out / complete_out: request r's token t at row hit_off[r] + t / tok_off[r] + t
 *       of R bytes ([sum T_hit][P][Rp] / [sum T_all][P][Rp], requests in order)
 *   block tables: one int32 array, request r's nblk entries at blk_off[r] (requests
 *       packed back to back in order); one table serves every layer and plane.
 *
 * Partial blocks: the scatter writes only slots t < T_all; later slots of the last
 * block keep their bytes.  Objects always carry whole blocks (fixed object size
 * B*Rp), so a partial block's object carries whatever those slots hold.
 *
 * Alignment: Rp, every stride and every buffer address must be multiples of 16 bytes.
 * Size: Rp, and R for kvl_slice_layer, at most 32 KiB (one shared-memory stage).
 * Aliasing: sources, pool, objects and outputs must not overlap (undefined otherwise);
 * with an injective block table every destination byte has exactly one writer.
 *
 * A plan records the request array and block tables it was built from; a call that
 * passes other arrays with that plan is refused on the device (KVL_EINVAL).
 *
 * Errors: problems the host can see (null or misaligned arguments, a bad geometry,
 * a layer outside [0, L), a plan too small) are returned at once and nothing is
 * launched.  Problems only the device can see (negative counts, misaligned request
 * fields, block ids out of range, duplicate block ids) are recorded in the plan's
 * status word: the offending work is skipped, nothing traps, and every later call
 * made with that plan does nothing until the plan is rebuilt.  Of the call that meets
 * the problem, any part of its other work may be left undone (its CTAs stop once they
 * see the status).  kvl_read_status reads the word back.  KVL_ECUDA reports a failed
 * launch.
 */
#ifndef KVL_H
#define KVL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t kvl_status;

#define KVL_OK 0
#define KVL_EINVAL 1 /* bad argument or geometry, negative count, null pointer */
#define KVL_EALIGN 2 /* pointer, stride or Rp not a multiple of 16 bytes */
#define KVL_ERANGE 3 /* block id outside the pool / source, or plan capacity exceeded */
#define KVL_EDUP 4   /* a pool block id used twice (only with check_injective) */
#define KVL_ECUDA 5  /* a CUDA launch or copy failed */
#define KVL_ETIMEOUT 6 /* a copy kernel's bounded wait on its own copies ran out (detail = CTA) */

#define KVL_GATHER 0      /* kvl_gather_layer_objects: pool -> objects */
#define KVL_SCATTER_BACK 1 /* kvl_gather_layer_objects: objects -> pool */

/* Geometry shared by every request of a batch (host memory). */
typedef struct kvl_geom {
    int32_t n_layers;        /* L */
    int32_t n_planes;        /* P: 2 = K,V planes; 1 = latent vector */
    int32_t block_tokens;    /* B: tokens per paged block */
    int32_t plane_row_bytes; /* Rp: bytes per token per plane, multiple of 16 */
    int64_t pool_blocks;     /* N: physical blocks in the pool */
} kvl_geom;

/* Launch options of a copy call (host memory; NULL = defaults). */
typedef struct kvl_launch {
    int32_t max_ctas; /* 0: one CTA on every SM (the whole GPU); k > 0: at most k CTAs,
                         i.e. the copy occupies at most k SMs and leaves the rest to
                         concurrent work (an I/O SM budget, as Tutti 阅读笔记 设计二
                         gives its I/O kernels a fixed SM partition) */
    int32_t flags;    /* 0, or KVL_LAUNCH_HOST_SRC or KVL_LAUNCH_HOST_DST (not both),
                         optionally OR KVL_LAUNCH_OVERLAP_PREVIOUS, KVL_LAUNCH_SHARE_SMS
                         and / or KVL_LAUNCH_PLAN_READY */
} kvl_launch;

/* The copy's sources (resp. destinations) are pinned host memory mapped into the
 * device address space (cudaHostAlloc / cudaHostRegister): e.g. DualPath's host
 * buffers, the full prompt KV held in Grace memory (DualPath KV Loading, "Dual-Path
 * Loading": pe_buffer / de_buffer and the final H2D into the HBM cache).  That side
 * is read (written) with ordinary 16-byte SM loads (stores) over NVLink-C2C; the HBM
 * side keeps the bulk-copy path.  Without the flag every buffer must be device memory. */
#define KVL_LAUNCH_HOST_SRC 1
#define KVL_LAUNCH_HOST_DST 2

/* The call may start copying before the kernel enqueued just before it on the stream
 * has finished, on the SMs that kernel has already left; it still finishes only after
 * that kernel has (so a later call without the flag sees both complete).  Meant for
 * the layer-wise pipeline's consecutive launches of one op on successive layers
 * (Tutti 阅读笔记, 伪代码 1: one I/O launch per layer; layers touch disjoint pool
 * regions), so that one launch's ramp-up fills the previous launch's tail.
 * The caller guarantees that the call touches no byte that the kernels it may overlap
 * write, and writes no byte that they read: the kernel just before it and, when that
 * call carried the flag too, the kernels that call may overlap in turn.  Reads of the
 * same plan, requests and tables are fine, but the plan's own kernels write the plan:
 * the first copy call after kvl_batch_plan must not carry the flag.  A call for the same plan, layer and op as
 * the kernel before it must not carry the flag (the two would share a work counter).
 * A call that overlaps a failing one may still copy: the failure shows in the plan's
 * status (kvl_read_status) once both have finished. */
#define KVL_LAUNCH_OVERLAP_PREVIOUS 4

/* Performance hint: the call's CTAs take half of an SM's shared memory (a 96 KiB
 * pipeline instead of 192 KiB), so that a CTA of the next launch, if that one carries
 * KVL_LAUNCH_OVERLAP_PREVIOUS, can run beside it on the same SM.  Set it on the call
 * just before a run of overlapping calls; KVL_LAUNCH_OVERLAP_PREVIOUS implies it.  A
 * call that runs alone is faster without it.  The host-memory variants ignore it. */
#define KVL_LAUNCH_SHARE_SMS 8

/* The caller declares that the plan (and the request array and tables it was built
 * from) was complete before the kernel enqueued just before this call began: no
 * kernel that may still run writes it, other than the copy calls' own claim counters
 * and status word.  True of every copy call of a layer-wise pipeline except the first
 * one after kvl_batch_plan.  A call that must wait for the kernel before it (no
 * KVL_LAUNCH_OVERLAP_PREVIOUS) then checks the plan, reads and decodes its first work
 * items and prefetches their source rows into L2 (cp.async.bulk.prefetch) while that
 * kernel drains, and waits only before its first copy; L2 is the device's point of
 * coherence, so rows the previous kernel writes are still read as it leaves them.
 * Results are the same with or without the flag; with a plan that is not complete,
 * undefined.  Ignored with KVL_LAUNCH_OVERLAP_PREVIOUS and by the host-memory
 * variants. */
#define KVL_LAUNCH_PLAN_READY 16

/* One request (device memory: the calls take an array of these in device memory).
 * All strides are in bytes. */
typedef struct kvl_request {
    const void *hit_src;          /* full block of the hit prefix (NULL if t_hit == 0) */
    const int32_t *hit_src_table; /* NULL, or nsrc full-block ids (device memory) */
    int64_t hit_src_blocks;       /* full blocks present at hit_src (bounds the ids) */
    int64_t hit_block_stride;
    int64_t hit_token_stride;
    int64_t hit_layer_stride;
    const void *miss_src;         /* miss KV (NULL if t_miss == 0) */
    int64_t miss_token_stride;
    int64_t miss_layer_stride;
    void *objects;                /* this request's K/V objects (NULL if never gathered) */
    int64_t obj_layer_stride;
    int64_t obj_plane_stride;
    int64_t obj_block_stride;
    int32_t t_hit;
    int32_t t_miss;
} kvl_request;

/* Bytes of device memory a plan for n_req requests in this geometry needs (0 for a
 * bad geometry).  The plan holds at most pool_blocks work items (injective tables
 * never need more), a 128-byte record per item and a claim counter per (layer, op). */
size_t kvl_plan_bytes(const kvl_geom *geom, int32_t n_req);

/* Plan layout, for callers that read the plan's arrays (byte offsets into the plan):
 * off[0] header, off[1] tok_off (int64[n_req+1]), off[2] hit_off (int64[n_req+1]),
 * off[3] blk_off (int64[n_req+1]), off[4] item_req (int32[pool_blocks]),
 * off[5] item_blk (int32[pool_blocks]), off[6] item records (always at byte 256),
 * off[7] claim counters, off[8] injectivity bitmap (the last section), off[9] total
 * bytes, off[10] tensor maps (6 x 128 bytes per request, starting at the first
 * 128-byte boundary at or after the plan's address + off[10], then an int32 of map
 * flags per request).  Sections are not
 * placed in index order.  The header's first int32 is the status and its int64 at
 * byte 16 the item count. */
void kvl_plan_layout(const kvl_geom *geom, int32_t n_req, size_t off[11]);

/* kvl_batch_plan -- the batch's work list, built on the device.
 * Computes exclusive prefix sums over requests of T_all (tok_off), T_hit (hit_off)
 * and nblk (blk_off), and the work list item i = blk_off[r] + j -> (r, j) for every
 * logical block j < nblk(r): the per-(request, block) items every later call walks,
 * so one launch per layer covers the whole batch (Tutti 阅读笔记, 伪代码 1
 * retrieve_layer and the note after it: the CPU launches the I/O kernel once per
 * layer, O(L) not O(L x blocks)).  Validates each request (counts >= 0, required
 * pointers non-null, 16-byte alignment), every pool block id (in [0, N)), every
 * full-block id of a hit block (in [0, hit_src_blocks)) and, if check_injective,
 * that no pool block id repeats.
 * The plan also describes each request's strided row sources (hit rows, miss rows)
 * by tensor maps, built on the device from templates that the host encodes with the
 * driver's cuTensorMapEncodeTiled (looked up through the runtime on the first plan
 * call; host work only, nothing allocated), when their strides lay the rows out
 * without overlap (each stride at least the extent below it) and some dimension spans
 * at least 1 MiB; the copy
 * calls then read a segment of rows of one source (a whole segment, or the rows a
 * block has left after its whole segments) with one tiled bulk-tensor load instead
 * of one bulk load per row.  The maps span exactly the rows a request
 * declares: T_hit rows of a full block without a table, all B token rows of each
 * of the hit_src_blocks blocks with a table (so with a table every one of those
 * blocks must be whole), and T_miss rows of the miss KV, each over all L layers.
 * Sources without maps (or a driver without the encoder) are read one bulk load per
 * row: the results are the same bytes either way.
 *   geom            host pointer
 *   d_reqs          device array of n_req requests (caller-owned, read only; may be
 *                   NULL when n_req == 0)
 *   d_block_tables  device int32 tables, packed in request order (read only; may be
 *                   NULL when n_req == 0)
 *   d_plan          device buffer of plan_bytes >= kvl_plan_bytes(geom, n_req) bytes,
 *                   16-byte aligned, caller-owned; overwritten.  The plan resolves
 *                   every item's addresses and block ids when it is built: later
 *                   edits to the requests or tables take effect only through a new
 *                   plan.  The copy calls update the plan's claim counters, so two
 *                   calls on one plan for the same layer and op must not overlap on
 *                   the GPU (calls for different layers or ops may).
 * Device-side status: EINVAL (detail = first bad request), EALIGN (detail = first bad
 * request), ERANGE (detail = smallest bad work item, or the item count when it
 * exceeds N), EDUP (detail = smallest repeated block id).  The largest code wins. */
kvl_status kvl_batch_plan(const kvl_geom *geom, int32_t n_req, const kvl_request *d_reqs,
                          const int32_t *d_block_tables, int32_t check_injective,
                          void *d_plan, size_t plan_bytes, void *stream);

/* kvl_batch_plan_static_scratch -- kvl_batch_plan for callers that cannot allocate
 * device memory.  The pages have no counterpart to this call.
 * Some callers cannot call cudaMalloc: for instance an inference engine whose own
 * allocator owns all of the HBM (its KV pool took it up front), where an extra
 * scratch allocation would fail or break the engine's accounting.  This call needs
 * no scratch from the caller: the injectivity bitmap lives in a fixed device array
 * inside libkvl.so (KVL_STATIC_SCRATCH_POOL_BLOCKS / 8 bytes = 512 KiB, held by
 * every GPU that loads the library until the process exits).  The caller still
 * passes the requests, the block tables and the plan, and the plan needs only
 * kvl_plan_layout(...)[8] bytes (everything before the bitmap section); the plan it
 * writes is the same as kvl_batch_plan's and the copy calls accept it.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * The array's device address belongs to the CUDA context the library's module was
 * loaded into.  Every call that is not being captured into a graph looks it up again
 * (cudaGetSymbolAddress, with the device current) and remembers it with the current
 * context's id; a call made while `stream` is capturing uses that remembered address
 * only if the current context is the one it was taken in, and otherwise returns
 * KVL_ECUDA with nothing launched.  So make one call on the device, outside capture,
 * before capturing one, and again after a cudaDeviceReset or a context switch.
 * Limits and sharing: pool_blocks above KVL_STATIC_SCRATCH_POOL_BLOCKS returns
 * KVL_EINVAL and launches nothing.  Every call on a device shares the one array,
 * which keeps the last call's contents; each call clears the bits it uses before
 * using them.  Calls that overlap on the GPU (other streams, other host threads)
 * race on the array in both directions: one call's bits can make another report a
 * duplicate that is not there, and one call's clearing can erase another's bits, so
 * a real duplicate can pass with KVL_OK and the copy calls would then give one pool
 * block two writers.  Serialise such calls.  Other arguments, checks and status
 * codes are those of kvl_batch_plan. */
#define KVL_STATIC_SCRATCH_POOL_BLOCKS (1 << 22)
kvl_status kvl_batch_plan_static_scratch(const kvl_geom *geom, int32_t n_req,
                                         const kvl_request *d_reqs, const int32_t *d_block_tables,
                                         int32_t check_injective, void *d_plan, size_t plan_bytes,
                                         void *stream);

/* The copy calls below work on the layers [layer, layer + layer_count) in one launch:
 * layer_count = 1 is the layer-wise pipeline of the pages (one launch per layer, as
 * soon as that layer's data exists); a larger count serves callers that have several
 * layers ready, e.g. restoring a whole prefix (Tutti 阅读笔记, 伪代码 1 and its note:
 * the I/O kernel is loaded once per layer, O(L) launches, not O(L x blocks)).
 * layer >= 0, layer_count >= 1, layer + layer_count <= L, pool_blocks * layer_count
 * < 2^31; otherwise KVL_EINVAL.  `launch` may be NULL (the whole GPU, no flags); a
 * negative max_ctas, an unknown flag or both host flags together is KVL_EINVAL.
 * d_plan is a plan built for this geom, and plan_bytes the size of the buffer at d_plan
 * (the plan_bytes the plan was built with, or the bytes a static-scratch plan needs).
 * plan_bytes below kvl_plan_layout(geom, 0)[8], the smallest plan of this geometry,
 * returns KVL_EINVAL and launches nothing, so no kernel reads past a buffer the host
 * knows to be too small.  The kernels read nothing of the plan beyond plan_bytes: a
 * plan whose recorded request count needs more than plan_bytes (a buffer sized for
 * fewer requests than the plan in it holds), or that was built for other arrays or
 * another geometry (L, P, B, Rp or N), is refused on the device (KVL_EINVAL in its
 * status) before any of its n_req-sized sections is read.
 * d_reqs and d_block_tables are the arrays the plan was built from; NULL only if it was
 * built from NULL (a batch of no requests); other NULLs are refused on the device. */

/* kvl_slice_layer -- hit_layer[l] = hit_full_block[:, l] for every request
 * (DualPath KV Loading, "Dual-Path Loading": objects table and the slice_layer step
 * of pe_read_path / de_read_path).  Writes, for each layer of the launch, sum(T_hit)
 * rows of R bytes to d_hit_out (device, caller-owned): launch layer i (= l - layer) at
 * row i*sum(T_hit) + hit_off[r] + t. */
kvl_status kvl_slice_layer(const kvl_geom *geom, const void *d_plan, size_t plan_bytes,
                           const kvl_request *d_reqs, int32_t layer, int32_t layer_count,
                           void *d_hit_out, const kvl_launch *launch, void *stream);

/* kvl_merge_scatter_paged -- slice, concatenate and scatter in one pass:
 * complete_layer[l] = hit_layer[l] rows then miss_layer[l] rows (DualPath KV Loading,
 * pe_read_path concatenate_tokens; de_read_path merge_layer), and token t of plane p
 * goes to pool block table[t / B], slot t % B (Tutti 阅读笔记, 前置知识 3, eq. (2)).
 *   d_pool          device pool [L][P][N][B][Rp], caller-owned; the slots of the
 *                   launch's layers named by the tables are written
 *   d_complete_out  NULL, or device memory that also receives complete_layer[l]:
 *                   launch layer i at row i*sum(T_all) + tok_off[r] + t, R bytes each */
kvl_status kvl_merge_scatter_paged(const kvl_geom *geom, const void *d_plan, size_t plan_bytes,
                                   const kvl_request *d_reqs, const int32_t *d_block_tables,
                                   int32_t layer, int32_t layer_count, void *d_pool,
                                   void *d_complete_out, const kvl_launch *launch, void *stream);

/* kvl_gather_layer_objects -- per-layer K/V objects <-> paged blocks.
 * direction KVL_GATHER: object (l, p, j) = pool block table[j] of plane p, layer l,
 * for every request: the 2*nblk objects of a layer ready for transfer (Tutti
 * 阅读笔记, 前置知识 5 eq. (4); the worked trace's 8,000 per-layer entries for 4,000
 * blocks).  direction KVL_SCATTER_BACK: the inverse, restoring objects into their
 * paged blocks (伪代码 1 retrieve_layer).  Each request's `objects` must be non-NULL. */
kvl_status kvl_gather_layer_objects(const kvl_geom *geom, const void *d_plan, size_t plan_bytes,
                                    const kvl_request *d_reqs, const int32_t *d_block_tables,
                                    int32_t layer, int32_t layer_count, void *d_pool,
                                    int32_t direction, const kvl_launch *launch, void *stream);

/* kvl_read_status -- copy the plan's status word and its detail to the host.
 * Synchronises `stream` first, so it reports every call enqueued before it.
 * code/detail may be NULL.  Returns KVL_ECUDA if the copy fails, else KVL_OK. */
kvl_status kvl_read_status(const void *d_plan, int32_t *code, int64_t *detail, void *stream);

/* kvl_diag_wait_timeout -- exercise the copy kernels' bounded wait.  Launches one
 * warp that waits, with the same bounded mbarrier wait the copy kernels use, for 16
 * bytes that nothing delivers; after limit_us microseconds (1 .. 10^7) it gives up and
 * writes KVL_ETIMEOUT to *d_status (device int32), then releases the barrier itself.
 * It copies nothing.  Used to check that a wait that runs out returns an error the
 * host can read and leaves the context usable. */
kvl_status kvl_diag_wait_timeout(int32_t limit_us, int32_t *d_status, void *stream);

/* Human-readable name of a status code (static string). */
const char *kvl_status_string(kvl_status s);

/* Kernel launches one call of each entry point makes (for launch accounting):
 * which = 0 plan, 1 slice, 2 merge-scatter, 3 gather / scatter-back. */
int32_t kvl_launches_per_call(int32_t which);

#ifdef __cplusplus
}
#endif

#endif /* KVL_H */

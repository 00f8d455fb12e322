/*
 * kvl_static_scratch_reset.c -- kvl_batch_plan_static_scratch across a context reset
 * and under stream capture, from plain C (no Python or torch, whose allocator would
 * not survive a cudaDeviceReset).
 *
 * Test infrastructure only.  Build (see tests/test_c_abi_program.py):
 *   cc -O1 -I include -I <cuda>/include tests/c_abi/kvl_static_scratch_reset.c
 *      -L <libkvl dir> -lkvl -L <cuda>/lib64 -lcudart -o kvl_static_scratch_reset
 * Exit status 0 and the line "static-scratch-reset: ok" when every check holds.
 *
 * The static-scratch plan builder keeps its bitmap in a device array inside the
 * library; that array's address belongs to the context the library's module was
 * loaded into, and cudaDeviceReset ends that context.  The program checks, on one
 * clean batch and one with a duplicate pool block id:
 *   1. before the reset: two calls in a row give the plan kvl_batch_plan gives
 *      (every byte below the bitmap section) and the same status;
 *   2. the same under stream capture (the captured graph, replayed, writes that plan);
 *   3. after cudaDeviceReset, a call made under capture before any call outside
 *      capture is refused with KVL_ECUDA and launches nothing (checked only when the
 *      new context's id differs from the old one, which is what the library keys on);
 *   4. after the reset, calls outside capture and then under capture again give
 *      kvl_batch_plan's plan, and a merge-scatter through the static-scratch plan
 *      equals one through kvl_batch_plan's (the copy kernels' shared-memory attribute
 *      belongs to the new context too).
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "kvl.h"

enum { NREQ = 3, L = 2, P = 2, B = 4, RP = 32, NPOOL = 64 };

static int failures = 0;

#define CUDA_OK(x)                                                                 \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
            exit(2);                                                               \
        }                                                                          \
    } while (0)

#define EXPECT(cond, ...)                                                          \
    do {                                                                           \
        if (!(cond)) {                                                             \
            fprintf(stderr, "line %d: ", __LINE__);                                \
            fprintf(stderr, __VA_ARGS__);                                          \
            fprintf(stderr, "\n");                                                 \
            failures++;                                                            \
        }                                                                          \
    } while (0)

static unsigned long long context_id(void)
{
    void *p = NULL, *q = NULL;
    enum cudaDriverEntryPointQueryResult r1, r2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &r1) !=
            cudaSuccess || r1 != cudaDriverEntryPointSuccess)
        return 0;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) !=
            cudaSuccess || r2 != cudaDriverEntryPointSuccess)
        return 0;
    CUcontext ctx = NULL;
    unsigned long long id = 0;
    if (((PFN_cuCtxGetCurrent_v4000)p)(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (((PFN_cuCtxGetId_v12000)q)(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

/* One batch in device memory: three requests, contiguous full blocks [T_hit, L, P, Rp]
 * and layer-major miss rows, one pool table (optionally with a repeated id). */
typedef struct {
    kvl_geom geom;
    kvl_request *d_reqs;
    int32_t *d_tables;
    uint8_t *d_hit, *d_miss, *d_pool_a, *d_pool_b;
    uint8_t *d_plan_ref, *d_plan_s;
    size_t ref_bytes, s_bytes, pool_bytes;
} batch;

static const int32_t t_hit[NREQ] = {40, 0, 23}, t_miss[NREQ] = {7, 12, 0};

static void make_batch(batch *b, int dup)
{
    const int64_t R = P * RP;
    b->geom.n_layers = L;
    b->geom.n_planes = P;
    b->geom.block_tokens = B;
    b->geom.plane_row_bytes = RP;
    b->geom.pool_blocks = NPOOL;
    int64_t hit_rows = 0, miss_rows = 0, nblk = 0;
    for (int r = 0; r < NREQ; r++) {
        hit_rows += t_hit[r];
        miss_rows += t_miss[r];
        nblk += (t_hit[r] + t_miss[r] + B - 1) / B;
    }
    int32_t *tables = malloc((size_t)nblk * 4);
    for (int64_t j = 0; j < nblk; j++) tables[j] = (int32_t)((j * 37 + 5) % NPOOL);
    if (dup) tables[9] = tables[3];
    size_t hit_bytes = (size_t)(hit_rows * L * R), miss_bytes = (size_t)(miss_rows * L * R);
    uint8_t *hbuf = malloc(hit_bytes), *mbuf = malloc(miss_bytes);
    for (size_t i = 0; i < hit_bytes; i++) hbuf[i] = (uint8_t)(i * 131 + 7);
    for (size_t i = 0; i < miss_bytes; i++) mbuf[i] = (uint8_t)(i * 71 + 3);
    CUDA_OK(cudaMalloc((void **)&b->d_hit, hit_bytes));
    CUDA_OK(cudaMalloc((void **)&b->d_miss, miss_bytes));
    CUDA_OK(cudaMalloc((void **)&b->d_tables, (size_t)nblk * 4));
    CUDA_OK(cudaMemcpy(b->d_hit, hbuf, hit_bytes, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(b->d_miss, mbuf, miss_bytes, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(b->d_tables, tables, (size_t)nblk * 4, cudaMemcpyHostToDevice));
    kvl_request reqs[NREQ];
    memset(reqs, 0, sizeof reqs);
    int64_t ho = 0, mo = 0;
    for (int r = 0; r < NREQ; r++) {
        kvl_request *q = &reqs[r];
        q->t_hit = t_hit[r];
        q->t_miss = t_miss[r];
        q->hit_src = t_hit[r] ? b->d_hit + ho * L * R : NULL;
        q->hit_src_blocks = (t_hit[r] + B - 1) / B;
        q->hit_block_stride = B * L * R;
        q->hit_token_stride = L * R;
        q->hit_layer_stride = R;
        q->miss_src = t_miss[r] ? b->d_miss + mo * L * R : NULL;
        q->miss_token_stride = R;
        q->miss_layer_stride = t_miss[r] * R;
        ho += t_hit[r];
        mo += t_miss[r];
    }
    CUDA_OK(cudaMalloc((void **)&b->d_reqs, sizeof reqs));
    CUDA_OK(cudaMemcpy(b->d_reqs, reqs, sizeof reqs, cudaMemcpyHostToDevice));
    size_t off[11];
    kvl_plan_layout(&b->geom, NREQ, off);
    b->ref_bytes = kvl_plan_bytes(&b->geom, NREQ);
    b->s_bytes = off[8];
    CUDA_OK(cudaMalloc((void **)&b->d_plan_ref, b->ref_bytes));
    CUDA_OK(cudaMalloc((void **)&b->d_plan_s, b->s_bytes));
    b->pool_bytes = (size_t)L * P * NPOOL * B * RP;
    CUDA_OK(cudaMalloc((void **)&b->d_pool_a, b->pool_bytes));
    CUDA_OK(cudaMalloc((void **)&b->d_pool_b, b->pool_bytes));
    free(tables);
    free(hbuf);
    free(mbuf);
}

static void free_batch(batch *b)
{
    void *p[] = {b->d_reqs, b->d_tables, b->d_hit, b->d_miss, b->d_pool_a, b->d_pool_b,
                 b->d_plan_ref, b->d_plan_s};
    for (size_t i = 0; i < sizeof p / sizeof p[0]; i++) CUDA_OK(cudaFree(p[i]));
}

/* The static-scratch plan (written just now) against kvl_batch_plan's: status and
 * every byte below the bitmap section (both buffers were zeroed before). */
static void compare_plans(const char *what, batch *b, cudaStream_t s)
{
    int32_t c1 = -1, c2 = -2;
    int64_t d1 = -1, d2 = -2;
    EXPECT(kvl_read_status(b->d_plan_ref, &c1, &d1, s) == KVL_OK, "%s: read status", what);
    EXPECT(kvl_read_status(b->d_plan_s, &c2, &d2, s) == KVL_OK, "%s: read status", what);
    EXPECT(c1 == c2 && d1 == d2, "%s: status %d/%lld vs %d/%lld", what, (int)c2, (long long)d2,
           (int)c1, (long long)d1);
    uint8_t *h1 = malloc(b->s_bytes), *h2 = malloc(b->s_bytes);
    CUDA_OK(cudaMemcpy(h1, b->d_plan_ref, b->s_bytes, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(h2, b->d_plan_s, b->s_bytes, cudaMemcpyDeviceToHost));
    EXPECT(memcmp(h1, h2, b->s_bytes) == 0, "%s: plans differ", what);
    free(h1);
    free(h2);
}

static void reference_plan(batch *b, cudaStream_t s)
{
    CUDA_OK(cudaMemsetAsync(b->d_plan_ref, 0, b->ref_bytes, s));
    EXPECT(kvl_batch_plan(&b->geom, NREQ, b->d_reqs, b->d_tables, 1, b->d_plan_ref, b->ref_bytes,
                          s) == KVL_OK, "kvl_batch_plan");
}

static kvl_status static_plan(batch *b, cudaStream_t s)
{
    return kvl_batch_plan_static_scratch(&b->geom, NREQ, b->d_reqs, b->d_tables, 1, b->d_plan_s,
                                         b->s_bytes, s);
}

/* Two calls in a row outside capture, then one captured into a graph and replayed. */
static void run_checks(const char *phase, int dup, cudaStream_t s)
{
    char what[96];
    batch b;
    make_batch(&b, dup);
    reference_plan(&b, s);
    for (int call = 0; call < 2; call++) {
        CUDA_OK(cudaMemsetAsync(b.d_plan_s, 0, b.s_bytes, s));
        EXPECT(static_plan(&b, s) == KVL_OK, "%s: static plan call %d", phase, call);
        snprintf(what, sizeof what, "%s, %s batch, call %d", phase, dup ? "duplicate" : "clean", call);
        compare_plans(what, &b, s);
    }
    CUDA_OK(cudaMemsetAsync(b.d_plan_s, 0, b.s_bytes, s));
    CUDA_OK(cudaStreamSynchronize(s));
    cudaGraph_t graph;
    cudaGraphExec_t exec;
    CUDA_OK(cudaStreamBeginCapture(s, cudaStreamCaptureModeGlobal));
    const kvl_status st = static_plan(&b, s);
    CUDA_OK(cudaStreamEndCapture(s, &graph));
    EXPECT(st == KVL_OK, "%s: static plan under capture: %d", phase, (int)st);
    CUDA_OK(cudaGraphInstantiate(&exec, graph, 0));
    CUDA_OK(cudaGraphLaunch(exec, s));
    snprintf(what, sizeof what, "%s, %s batch, captured", phase, dup ? "duplicate" : "clean");
    compare_plans(what, &b, s);
    CUDA_OK(cudaGraphExecDestroy(exec));
    CUDA_OK(cudaGraphDestroy(graph));
    if (!dup) {
        /* the copy kernels take the static-scratch plan like kvl_batch_plan's */
        CUDA_OK(cudaMemsetAsync(b.d_pool_a, 0xA5, b.pool_bytes, s));
        CUDA_OK(cudaMemsetAsync(b.d_pool_b, 0xA5, b.pool_bytes, s));
        for (int l = 0; l < L; l++) {
            EXPECT(kvl_merge_scatter_paged(&b.geom, b.d_plan_ref, b.ref_bytes, b.d_reqs, b.d_tables,
                                           l, 1, b.d_pool_a, NULL, NULL, s) == KVL_OK, "merge ref");
            EXPECT(kvl_merge_scatter_paged(&b.geom, b.d_plan_s, b.s_bytes, b.d_reqs, b.d_tables, l,
                                           1, b.d_pool_b, NULL, NULL, s) == KVL_OK, "merge static");
        }
        uint8_t *pa = malloc(b.pool_bytes), *pb = malloc(b.pool_bytes);
        CUDA_OK(cudaStreamSynchronize(s));
        CUDA_OK(cudaMemcpy(pa, b.d_pool_a, b.pool_bytes, cudaMemcpyDeviceToHost));
        CUDA_OK(cudaMemcpy(pb, b.d_pool_b, b.pool_bytes, cudaMemcpyDeviceToHost));
        EXPECT(memcmp(pa, pb, b.pool_bytes) == 0, "%s: pools differ", phase);
        size_t written = 0;
        for (size_t i = 0; i < b.pool_bytes; i++) written += pa[i] != 0xA5;
        EXPECT(written > 0, "%s: merge-scatter wrote nothing", phase);
        int32_t code = -1;
        int64_t detail = -1;
        EXPECT(kvl_read_status(b.d_plan_s, &code, &detail, s) == KVL_OK && code == KVL_OK,
               "%s: status after merge-scatter %d", phase, (int)code);
        free(pa);
        free(pb);
    }
    free_batch(&b);
}

int main(void)
{
    CUDA_OK(cudaSetDevice(0));
    cudaStream_t s;
    CUDA_OK(cudaStreamCreate(&s));
    run_checks("before reset", 0, s);
    run_checks("before reset", 1, s);
    const unsigned long long old_id = context_id();
    CUDA_OK(cudaStreamDestroy(s));

    CUDA_OK(cudaDeviceReset());
    CUDA_OK(cudaSetDevice(0));
    CUDA_OK(cudaStreamCreate(&s));
    const unsigned long long new_id = context_id();
    if (old_id != 0 && new_id != 0 && old_id != new_id) {
        /* the remembered address belongs to the old context: a captured call refuses */
        batch b;
        make_batch(&b, 0);
        CUDA_OK(cudaMemset(b.d_plan_s, 0x5A, b.s_bytes));
        CUDA_OK(cudaDeviceSynchronize());
        cudaGraph_t graph;
        CUDA_OK(cudaStreamBeginCapture(s, cudaStreamCaptureModeGlobal));
        const kvl_status st = static_plan(&b, s);
        CUDA_OK(cudaStreamEndCapture(s, &graph));
        EXPECT(st == KVL_ECUDA, "captured call after reset: %d, want KVL_ECUDA", (int)st);
        size_t nodes = 1;
        CUDA_OK(cudaGraphGetNodes(graph, NULL, &nodes));
        EXPECT(nodes == 0, "captured call after reset launched %zu kernels", nodes);
        CUDA_OK(cudaGraphDestroy(graph));
        free_batch(&b);
    } else {
        printf("context ids %llu -> %llu: the refusal under capture is not checked\n", old_id, new_id);
    }
    run_checks("after reset", 0, s);
    run_checks("after reset", 1, s);
    CUDA_OK(cudaStreamDestroy(s));
    if (failures) {
        fprintf(stderr, "static-scratch-reset: %d failures\n", failures);
        return 1;
    }
    printf("static-scratch-reset: ok\n");
    return 0;
}

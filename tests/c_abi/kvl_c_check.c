/*
 * kvl_c_check.c -- the C ABI used from plain C, with no Python or torch: device memory
 * from cudaMalloc, every call through include/kvl.h, every result compared byte for
 * byte with the CPU oracle (oracle/kvl_oracle.c, compiled into this test program).
 *
 * Test infrastructure only.  Build (see tests/test_c_abi_program.py):
 *   cc -O1 -I include -I <cuda>/include tests/c_abi/kvl_c_check.c oracle/kvl_oracle.c
 *      -L <libkvl dir> -lkvl -L <cuda>/lib64 -lcudart -o kvl_c_check
 * Exit status 0 and the line "c-abi: ok" when every comparison holds.
 *
 * Two batches of two requests each, over a shuffled pool table.  Request 0 reads its
 * hit prefix from shuffled full blocks (a full-block table) and writes layer-major
 * objects; request 1 reads a contiguous full block and writes block-major objects.
 * Layers 1 and up of each op run with KVL_LAUNCH_OVERLAP_PREVIOUS, layer 0 with
 * KVL_LAUNCH_SHARE_SMS; scatter-back restores every layer in one launch.
 *   - "small": L = 3, P = 2 planes of 48 bytes, B = 4; sources far below the span the
 *     plan's tensor maps need, so every row moves by its own bulk load;
 *   - "mapped": L = 3, P = 2 planes of 2 KiB, B = 16, hundreds of tokens; the hit and
 *     miss sources span megabytes, so whole segments go through the tensor maps.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "kvl.h"

/* The oracle's own types and entry points (oracle/kvl_oracle.c). */
typedef struct {
    int32_t L, P, B, Rp;
    int64_t n_pool;
} oracle_geom;

typedef struct {
    const uint8_t *hit_src;
    const int32_t *hit_src_table;
    int64_t hit_src_blocks;
    int64_t hit_block_stride, hit_token_stride, hit_layer_stride;
    const uint8_t *miss_src;
    int64_t miss_token_stride, miss_layer_stride;
    uint8_t *objects;
    int64_t obj_layer_stride, obj_plane_stride, obj_block_stride;
    int32_t t_hit, t_miss;
} oracle_req;

int oracle_slice_layer(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                       int32_t layer, uint8_t *hit_out);
int oracle_merge_scatter(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                         const int32_t *tables, int32_t layer, uint8_t *pool,
                         uint8_t *complete_out);
int oracle_gather_objects(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                          const int32_t *tables, int32_t layer, const uint8_t *pool);
int oracle_scatter_back(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                        const int32_t *tables, int32_t layer, uint8_t *pool);

enum { NREQ = 2, SENTINEL = 0xA5 };

static int failures = 0;

#define CUDA_OK(x)                                                                 \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
            exit(2);                                                               \
        }                                                                          \
    } while (0)

#define KVL_OK_(x)                                                                 \
    do {                                                                           \
        kvl_status s_ = (x);                                                       \
        if (s_ != KVL_OK) {                                                        \
            fprintf(stderr, "kvl status %d (%s) at line %d\n", (int)s_, kvl_status_string(s_), __LINE__); \
            exit(3);                                                               \
        }                                                                          \
    } while (0)

static void check_equal(const char *what, const uint8_t *dev, const uint8_t *want, size_t n)
{
    uint8_t *got = (uint8_t *)malloc(n ? n : 1);
    CUDA_OK(cudaMemcpy(got, dev, n, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < n; i++)
        if (got[i] != want[i]) {
            fprintf(stderr, "%s: byte %zu differs (%u, oracle %u)\n", what, i, got[i], want[i]);
            failures++;
            break;
        }
    free(got);
}

/* Deterministic payload bytes (a 64-bit linear congruential sequence). */
static void fill(uint8_t *p, size_t n, uint64_t seed)
{
    uint64_t x = seed;
    for (size_t i = 0; i < n; i++) {
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        p[i] = (uint8_t)(x >> 56);
    }
}

/* The first n entries of a seeded shuffle of 0 .. m-1 (injective). */
static void shuffled_ids(int32_t *out, int32_t n, int32_t m, uint64_t seed)
{
    int32_t *all = (int32_t *)malloc(sizeof(int32_t) * (size_t)(m ? m : 1));
    uint64_t x = seed;
    for (int32_t i = 0; i < m; i++) all[i] = i;
    for (int32_t i = m - 1; i > 0; i--) {
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        const int32_t j = (int32_t)((x >> 33) % (uint64_t)(i + 1));
        const int32_t t = all[i];
        all[i] = all[j];
        all[j] = t;
    }
    memcpy(out, all, sizeof(int32_t) * (size_t)n);
    free(all);
}

static void *dev_copy(const void *host, size_t n)
{
    void *d = NULL;
    CUDA_OK(cudaMalloc(&d, n ? n : 16));
    if (n) CUDA_OK(cudaMemcpy(d, host, n, cudaMemcpyHostToDevice));
    return d;
}

/* One batch of two requests through every entry point, checked against the oracle. */
static void run_batch(const char *name, int32_t L, int32_t P, int32_t B, int32_t RP,
                      const int32_t t_hit[NREQ], const int32_t t_miss[NREQ], uint64_t seed)
{
    const int64_t R = (int64_t)P * RP;
    int32_t nblk[NREQ], ntab = 0, n_hit = 0, n_all = 0;
    for (int r = 0; r < NREQ; r++) {
        nblk[r] = (t_hit[r] + t_miss[r] + B - 1) / B;
        ntab += nblk[r];
        n_hit += t_hit[r];
        n_all += t_hit[r] + t_miss[r];
    }
    const int32_t npool = ntab + ntab / 2 + 4;
    int32_t *tables = (int32_t *)malloc(sizeof(int32_t) * (size_t)ntab);
    shuffled_ids(tables, ntab, npool, seed);
    /* request 0: its hit prefix in nsrc shuffled full blocks [B][L][P][RP] out of
       nsrc + 1 stored */
    const int32_t nsrc = (t_hit[0] + B - 1) / B;
    const int64_t src_blocks = nsrc + 1, blk_bytes = (int64_t)B * L * R;
    int32_t *src_table = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nsrc ? nsrc : 1));
    shuffled_ids(src_table, nsrc, (int32_t)src_blocks, seed + 1);

    size_t hit0_n = (size_t)(src_blocks * blk_bytes), hit1_n = (size_t)t_hit[1] * L * R;
    size_t miss_n[NREQ] = {(size_t)L * t_miss[0] * R, (size_t)L * t_miss[1] * R};
    size_t obj_n[NREQ] = {(size_t)L * P * nblk[0] * B * RP, (size_t)L * P * nblk[1] * B * RP};
    size_t pool_n = (size_t)L * P * npool * B * RP;

    uint8_t *hit0 = malloc(hit0_n), *hit1 = malloc(hit1_n ? hit1_n : 1);
    uint8_t *miss0 = malloc(miss_n[0] ? miss_n[0] : 1), *miss1 = malloc(miss_n[1] ? miss_n[1] : 1);
    uint8_t *obj_h[NREQ] = {malloc(obj_n[0]), malloc(obj_n[1])};
    uint8_t *pool_h = malloc(pool_n);
    fill(hit0, hit0_n, seed + 2);
    fill(hit1, hit1_n, seed + 3);
    fill(miss0, miss_n[0], seed + 4);
    fill(miss1, miss_n[1], seed + 5);
    memset(obj_h[0], SENTINEL, obj_n[0]);
    memset(obj_h[1], SENTINEL, obj_n[1]);
    memset(pool_h, SENTINEL, pool_n);

    uint8_t *d_hit0 = dev_copy(hit0, hit0_n), *d_hit1 = dev_copy(hit1, hit1_n);
    uint8_t *d_miss0 = dev_copy(miss0, miss_n[0]), *d_miss1 = dev_copy(miss1, miss_n[1]);
    uint8_t *d_obj[NREQ] = {dev_copy(obj_h[0], obj_n[0]), dev_copy(obj_h[1], obj_n[1])};
    uint8_t *d_pool = dev_copy(pool_h, pool_n);
    int32_t *d_tables = dev_copy(tables, sizeof(int32_t) * (size_t)ntab);
    int32_t *d_src_table = dev_copy(src_table, sizeof(int32_t) * (size_t)nsrc);

    /* the same requests twice: device pointers for the library, host ones for the oracle */
    kvl_request req[NREQ];
    oracle_req oreq[NREQ];
    memset(req, 0, sizeof req);
    memset(oreq, 0, sizeof oreq);
    /* request 0: shuffled full blocks, miss layer-major [L][T_miss][P][RP], objects
       layer-major [L][P][nblk][B][RP] */
    req[0].hit_src = d_hit0;                  oreq[0].hit_src = hit0;
    req[0].hit_src_table = d_src_table;       oreq[0].hit_src_table = src_table;
    req[0].hit_src_blocks = oreq[0].hit_src_blocks = src_blocks;
    req[0].hit_block_stride = oreq[0].hit_block_stride = blk_bytes;
    req[0].hit_token_stride = oreq[0].hit_token_stride = (int64_t)L * R;
    req[0].hit_layer_stride = oreq[0].hit_layer_stride = R;
    req[0].miss_src = d_miss0;                oreq[0].miss_src = miss0;
    req[0].miss_token_stride = oreq[0].miss_token_stride = R;
    req[0].miss_layer_stride = oreq[0].miss_layer_stride = (int64_t)t_miss[0] * R;
    req[0].objects = d_obj[0];                oreq[0].objects = obj_h[0];
    req[0].obj_layer_stride = oreq[0].obj_layer_stride = (int64_t)P * nblk[0] * B * RP;
    req[0].obj_plane_stride = oreq[0].obj_plane_stride = (int64_t)nblk[0] * B * RP;
    req[0].obj_block_stride = oreq[0].obj_block_stride = (int64_t)B * RP;
    /* request 1: contiguous full block [T_hit][L][P][RP], miss token-major
       [T_miss][L][P][RP], objects block-major [nblk][L][P][B][RP] */
    req[1].hit_src = d_hit1;                  oreq[1].hit_src = hit1;
    req[1].hit_src_blocks = oreq[1].hit_src_blocks = (t_hit[1] + B - 1) / B;
    req[1].hit_block_stride = oreq[1].hit_block_stride = (int64_t)B * L * R;
    req[1].hit_token_stride = oreq[1].hit_token_stride = (int64_t)L * R;
    req[1].hit_layer_stride = oreq[1].hit_layer_stride = R;
    req[1].miss_src = d_miss1;                oreq[1].miss_src = miss1;
    req[1].miss_token_stride = oreq[1].miss_token_stride = (int64_t)L * R;
    req[1].miss_layer_stride = oreq[1].miss_layer_stride = R;
    req[1].objects = d_obj[1];                oreq[1].objects = obj_h[1];
    req[1].obj_layer_stride = oreq[1].obj_layer_stride = (int64_t)P * B * RP;
    req[1].obj_plane_stride = oreq[1].obj_plane_stride = (int64_t)B * RP;
    req[1].obj_block_stride = oreq[1].obj_block_stride = (int64_t)L * P * B * RP;
    for (int r = 0; r < NREQ; r++) {
        req[r].t_hit = oreq[r].t_hit = t_hit[r];
        req[r].t_miss = oreq[r].t_miss = t_miss[r];
    }
    kvl_request *d_reqs = dev_copy(req, sizeof req);

    const kvl_geom geom = {L, P, B, RP, npool};
    const oracle_geom og = {L, P, B, RP, npool};
    size_t plan_bytes = kvl_plan_bytes(&geom, NREQ);
    void *d_plan = NULL;
    CUDA_OK(cudaMalloc(&d_plan, plan_bytes));
    cudaStream_t s;
    CUDA_OK(cudaStreamCreate(&s));
    KVL_OK_(kvl_batch_plan(&geom, NREQ, d_reqs, d_tables, 1, d_plan, plan_bytes, s));

    /* per op, layer by layer: layer 0 leaves room on the SMs, layers 1.. overlap it */
    kvl_launch first = {0, KVL_LAUNCH_SHARE_SMS}, next = {0, KVL_LAUNCH_OVERLAP_PREVIOUS};
    uint8_t *d_hit_out = NULL, *d_complete = NULL;
    CUDA_OK(cudaMalloc((void **)&d_hit_out, (size_t)L * n_hit * R));
    CUDA_OK(cudaMalloc((void **)&d_complete, (size_t)L * n_all * R));
    for (int l = 0; l < L; l++)
        KVL_OK_(kvl_slice_layer(&geom, d_plan, plan_bytes, d_reqs, l, 1, d_hit_out + (size_t)l * n_hit * R,
                                l ? &next : &first, s));
    for (int l = 0; l < L; l++)
        KVL_OK_(kvl_merge_scatter_paged(&geom, d_plan, plan_bytes, d_reqs, d_tables, l, 1, d_pool,
                                        d_complete + (size_t)l * n_all * R, l ? &next : &first, s));
    for (int l = 0; l < L; l++)
        KVL_OK_(kvl_gather_layer_objects(&geom, d_plan, plan_bytes, d_reqs, d_tables, l, 1, d_pool,
                                         KVL_GATHER,
                                         l ? &next : &first, s));
    CUDA_OK(cudaStreamSynchronize(s));

    uint8_t *want_hit = malloc((size_t)n_hit * R), *want_complete = malloc((size_t)n_all * R);
    char what[96];
    for (int l = 0; l < L; l++) {
        if (oracle_slice_layer(&og, NREQ, oreq, l, want_hit) != 0) failures++;
        if (oracle_merge_scatter(&og, NREQ, oreq, tables, l, pool_h, want_complete) != 0) failures++;
        if (oracle_gather_objects(&og, NREQ, oreq, tables, l, pool_h) != 0) failures++;
        snprintf(what, sizeof what, "%s: hit_layer[%d]", name, l);
        check_equal(what, d_hit_out + (size_t)l * n_hit * R, want_hit, (size_t)n_hit * R);
        snprintf(what, sizeof what, "%s: complete_layer[%d]", name, l);
        check_equal(what, d_complete + (size_t)l * n_all * R, want_complete, (size_t)n_all * R);
    }
    snprintf(what, sizeof what, "%s: pool after merge-scatter", name);
    check_equal(what, d_pool, pool_h, pool_n);
    snprintf(what, sizeof what, "%s: objects of request 0", name);
    check_equal(what, d_obj[0], obj_h[0], obj_n[0]);
    snprintf(what, sizeof what, "%s: objects of request 1", name);
    check_equal(what, d_obj[1], obj_h[1], obj_n[1]);

    /* scatter back into a blank pool: all layers in one launch */
    memset(pool_h, SENTINEL, pool_n);
    CUDA_OK(cudaMemset(d_pool, SENTINEL, pool_n));
    KVL_OK_(kvl_gather_layer_objects(&geom, d_plan, plan_bytes, d_reqs, d_tables, 0, L, d_pool,
                                     KVL_SCATTER_BACK, NULL, s));
    for (int l = 0; l < L; l++)
        if (oracle_scatter_back(&og, NREQ, oreq, tables, l, pool_h) != 0) failures++;
    CUDA_OK(cudaStreamSynchronize(s));
    snprintf(what, sizeof what, "%s: pool after scatter-back", name);
    check_equal(what, d_pool, pool_h, pool_n);

    int32_t code = -1;
    int64_t detail = -1;
    KVL_OK_(kvl_read_status(d_plan, &code, &detail, s));
    if (code != KVL_OK) {
        fprintf(stderr, "%s: plan status %d detail %lld\n", name, (int)code, (long long)detail);
        failures++;
    }

    CUDA_OK(cudaStreamDestroy(s));
    void *dev[] = {d_hit0, d_hit1, d_miss0, d_miss1, d_obj[0], d_obj[1], d_pool, d_tables,
                   d_src_table, d_reqs, d_plan, d_hit_out, d_complete};
    for (size_t i = 0; i < sizeof dev / sizeof dev[0]; i++) CUDA_OK(cudaFree(dev[i]));
    void *host[] = {tables, src_table, hit0, hit1, miss0, miss1, obj_h[0], obj_h[1], pool_h,
                    want_hit, want_complete};
    for (size_t i = 0; i < sizeof host / sizeof host[0]; i++) free(host[i]);
}

int main(void)
{
    const int32_t small_hit[NREQ] = {9, 6}, small_miss[NREQ] = {2, 5};
    run_batch("small", 3, 2, 4, 48, small_hit, small_miss, 101);
    /* hit rows of 2 KiB planes, tokens 12 KiB apart: a source of 600 tokens spans 7 MB */
    const int32_t mapped_hit[NREQ] = {600, 700}, mapped_miss[NREQ] = {300, 90};
    run_batch("mapped", 3, 2, 16, 2048, mapped_hit, mapped_miss, 202);
    if (failures) {
        fprintf(stderr, "c-abi: %d failures\n", failures);
        return 1;
    }
    printf("c-abi: ok\n");
    return 0;
}

/*
 * kvl_c_check.c -- the C ABI used from plain C, with no Python or torch: device memory
 * from cudaMalloc, every call through include/kvl.h, every result compared byte for
 * byte with the CPU oracle (oracle/kvl_oracle.c, compiled into this test program).
 *
 * Test infrastructure only.  Build (see tests/test_gpu_c_abi.py):
 *   cc -O1 -I include -I <cuda>/include tests/c_abi/kvl_c_check.c oracle/kvl_oracle.c
 *      -L <libkvl dir> -lkvl -L <cuda>/lib64 -lcudart -o kvl_c_check
 * Exit status 0 and the line "c-abi: ok" when every comparison holds.
 *
 * Batch: two requests over L = 3 layers, P = 2 planes of 48 bytes, B = 4 tokens per
 * block, a shuffled pool table; request 0 reads its hit prefix from shuffled full
 * blocks (a full-block table), request 1 from a contiguous full block; the second
 * request's objects are block-major.  Layers 1 and 2 of each op run with
 * KVL_LAUNCH_OVERLAP_PREVIOUS, layer 0 with KVL_LAUNCH_SHARE_SMS.
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

enum { L = 3, P = 2, B = 4, RP = 48, R = P * RP, NREQ = 2, NPOOL = 16 };
enum { SENTINEL = 0xA5 };

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

static void *dev_copy(const void *host, size_t n)
{
    void *d = NULL;
    CUDA_OK(cudaMalloc(&d, n ? n : 16));
    if (n) CUDA_OK(cudaMemcpy(d, host, n, cudaMemcpyHostToDevice));
    return d;
}

int main(void)
{
    const int32_t t_hit[NREQ] = {9, 6}, t_miss[NREQ] = {2, 5};
    int32_t nblk[NREQ], ntab = 0, n_hit = 0, n_all = 0;
    for (int r = 0; r < NREQ; r++) {
        nblk[r] = (t_hit[r] + t_miss[r] + B - 1) / B;
        ntab += nblk[r];
        n_hit += t_hit[r];
        n_all += t_hit[r] + t_miss[r];
    }
    /* pool table: a fixed shuffle of the pool's block ids (injective) */
    const int32_t tables[] = {11, 3, 14, 0, 7, 9};
    if ((int)(sizeof tables / sizeof tables[0]) != ntab) return 4;
    /* request 0: hit prefix in 3 shuffled full blocks [B][L][P][RP] out of 4 stored */
    const int32_t src_table[] = {2, 0, 3};
    const int64_t src_blocks = 4, blk_bytes = (int64_t)B * L * R;

    size_t hit0_n = (size_t)(src_blocks * blk_bytes), hit1_n = (size_t)t_hit[1] * L * R;
    size_t miss_n[NREQ] = {(size_t)L * t_miss[0] * R, (size_t)L * t_miss[1] * R};
    size_t obj_n[NREQ] = {(size_t)L * P * nblk[0] * B * RP, (size_t)L * P * nblk[1] * B * RP};
    size_t pool_n = (size_t)L * P * NPOOL * B * RP;

    uint8_t *hit0 = malloc(hit0_n), *hit1 = malloc(hit1_n);
    uint8_t *miss0 = malloc(miss_n[0]), *miss1 = malloc(miss_n[1]);
    uint8_t *obj_h[NREQ] = {malloc(obj_n[0]), malloc(obj_n[1])};
    uint8_t *pool_h = malloc(pool_n);
    fill(hit0, hit0_n, 1);
    fill(hit1, hit1_n, 2);
    fill(miss0, miss_n[0], 3);
    fill(miss1, miss_n[1], 4);
    memset(obj_h[0], SENTINEL, obj_n[0]);
    memset(obj_h[1], SENTINEL, obj_n[1]);
    memset(pool_h, SENTINEL, pool_n);

    uint8_t *d_hit0 = dev_copy(hit0, hit0_n), *d_hit1 = dev_copy(hit1, hit1_n);
    uint8_t *d_miss0 = dev_copy(miss0, miss_n[0]), *d_miss1 = dev_copy(miss1, miss_n[1]);
    uint8_t *d_obj[NREQ] = {dev_copy(obj_h[0], obj_n[0]), dev_copy(obj_h[1], obj_n[1])};
    uint8_t *d_pool = dev_copy(pool_h, pool_n);
    int32_t *d_tables = dev_copy(tables, sizeof tables);
    int32_t *d_src_table = dev_copy(src_table, sizeof src_table);

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

    const kvl_geom geom = {L, P, B, RP, NPOOL};
    const oracle_geom og = {L, P, B, RP, NPOOL};
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
        KVL_OK_(kvl_slice_layer(&geom, d_plan, d_reqs, l, 1, d_hit_out + (size_t)l * n_hit * R,
                                l ? &next : &first, s));
    for (int l = 0; l < L; l++)
        KVL_OK_(kvl_merge_scatter_paged(&geom, d_plan, d_reqs, d_tables, l, 1, d_pool,
                                        d_complete + (size_t)l * n_all * R, l ? &next : &first, s));
    for (int l = 0; l < L; l++)
        KVL_OK_(kvl_gather_layer_objects(&geom, d_plan, d_reqs, d_tables, l, 1, d_pool, KVL_GATHER,
                                         l ? &next : &first, s));
    CUDA_OK(cudaStreamSynchronize(s));

    uint8_t *want_hit = malloc((size_t)n_hit * R), *want_complete = malloc((size_t)n_all * R);
    char what[64];
    for (int l = 0; l < L; l++) {
        if (oracle_slice_layer(&og, NREQ, oreq, l, want_hit) != 0) failures++;
        if (oracle_merge_scatter(&og, NREQ, oreq, tables, l, pool_h, want_complete) != 0) failures++;
        if (oracle_gather_objects(&og, NREQ, oreq, tables, l, pool_h) != 0) failures++;
        snprintf(what, sizeof what, "hit_layer[%d]", l);
        check_equal(what, d_hit_out + (size_t)l * n_hit * R, want_hit, (size_t)n_hit * R);
        snprintf(what, sizeof what, "complete_layer[%d]", l);
        check_equal(what, d_complete + (size_t)l * n_all * R, want_complete, (size_t)n_all * R);
    }
    check_equal("pool after merge-scatter", d_pool, pool_h, pool_n);
    check_equal("objects of request 0", d_obj[0], obj_h[0], obj_n[0]);
    check_equal("objects of request 1", d_obj[1], obj_h[1], obj_n[1]);

    /* scatter back into a blank pool: all layers in one launch */
    memset(pool_h, SENTINEL, pool_n);
    CUDA_OK(cudaMemset(d_pool, SENTINEL, pool_n));
    KVL_OK_(kvl_gather_layer_objects(&geom, d_plan, d_reqs, d_tables, 0, L, d_pool,
                                     KVL_SCATTER_BACK, NULL, s));
    for (int l = 0; l < L; l++)
        if (oracle_scatter_back(&og, NREQ, oreq, tables, l, pool_h) != 0) failures++;
    CUDA_OK(cudaStreamSynchronize(s));
    check_equal("pool after scatter-back", d_pool, pool_h, pool_n);

    int32_t code = -1;
    int64_t detail = -1;
    KVL_OK_(kvl_read_status(d_plan, &code, &detail, s));
    if (code != KVL_OK) {
        fprintf(stderr, "plan status %d detail %lld\n", (int)code, (long long)detail);
        failures++;
    }
    if (failures) {
        fprintf(stderr, "c-abi: %d failures\n", failures);
        return 1;
    }
    printf("c-abi: ok\n");
    return 0;
}

/*
 * kvl_oracle.c -- plain, slow, obviously correct CPU reference of the layer-wise
 * paged KV block reshuffle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no code,
 * header, helper or constant with the CUDA path, and it never calls it.
 *
 * What it computes, step by step in the pages' order:
 *
 *   slice_layer      hit_layer[l] = hit_full_block[:, l]
 *                    (DualPath KV Loading, "Dual-Path Loading": objects table,
 *                     hit_full_block [T_hit, L, C_KV] -> hit_layer[l] [T_hit, C_KV];
 *                     pe_read_path / de_read_path listings, slice_layer step)
 *   concatenate      complete_layer[l] = hit_layer[l] rows, then miss_layer[l] rows
 *                    (same page, concatenate_tokens(hit_layer, miss_layer) in
 *                     pe_read_path; merge_layer in de_read_path)
 *   scatter_paged    token t of plane p goes to pool block table[t / B], slot t % B
 *                    (Tutti 阅读笔记, 前置知识 3 "分页 KV 内存管理", eq. (2): a block is
 *                     [B_tokens, H, d]; a sequence's blocks are linked by a block table)
 *   gather_objects   one K object and one V object per (layer, block): object
 *                    (l, p, j) = pool block table[j] of plane p in layer l
 *                    (Tutti 阅读笔记, 前置知识 5, eqs. (3)(4); 设计一 §3.1 GPU file pool,
 *                     2L objects per block; 伪代码 1 retrieve_layer, one call per layer)
 *   scatter_back     the inverse of gather_objects (retrieve_layer restores objects
 *                    into the paged HBM blocks)
 *   plan             exclusive prefix sums over requests of T_all, T_hit and
 *                    ceil(T_all / B), and the (request, block) work list
 *
 * Layouts (all byte offsets; R = P * Rp):
 *   hit token t, layer l, plane p: hit_src + sb(t/B)*hit_block_stride
 *        + (t%B)*hit_token_stride + l*hit_layer_stride + p*Rp,
 *        sb(j) = hit_src_table ? hit_src_table[j] : j
 *   miss token t (T_hit <= t < T_all): miss_src + (t-T_hit)*miss_token_stride
 *        + l*miss_layer_stride + p*Rp
 *   pool block b, slot s:  pool + (((l*P + p)*N + b)*B + s)*Rp
 *   object (l, p, j):      objects + l*obj_layer_stride + p*obj_plane_stride
 *                          + j*obj_block_stride (layer-major [L][P][nblk][B][Rp], or
 *                          block-major [nblk][L][P][B][Rp]: one GPU file per block
 *                          holding its 2L objects, Tutti 阅读笔记 设计一 §3.1)
 *   hit_out / complete_out: row (prefix + t) of R bytes, requests packed in order
 *
 * Readings where the pages are silent: the pool is [L][P][N][B][Rp]; K is plane 0;
 * slots of a partial last block past T_all are not written by the scatter, and the
 * object of such a block carries the whole block, whatever those slots hold.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status values, as the library documents them (defined here independently). */
#define OR_OK 0
#define OR_EINVAL 1
#define OR_ERANGE 3
#define OR_EDUP 4

typedef struct {
    int32_t L, P, B, Rp;
    int64_t n_pool;
} oracle_geom;

typedef struct {
    const uint8_t *hit_src;
    const int32_t *hit_src_table;   /* NULL = the hit prefix is stored in order */
    int64_t hit_src_blocks;
    int64_t hit_block_stride, hit_token_stride, hit_layer_stride;
    const uint8_t *miss_src;
    int64_t miss_token_stride, miss_layer_stride;
    uint8_t *objects;
    int64_t obj_layer_stride, obj_plane_stride, obj_block_stride;
    int32_t t_hit, t_miss;
} oracle_req;

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

static int64_t t_all_of(const oracle_req *q) { return (int64_t)q->t_hit + q->t_miss; }

/* Row of hit token t in layer l (all P planes, R bytes), or NULL if its full
 * block id is out of range. */
static const uint8_t *hit_row(const oracle_geom *g, const oracle_req *q, int32_t l, int64_t t)
{
    int64_t j = t / g->B, s = t % g->B;
    int64_t blk = q->hit_src_table ? q->hit_src_table[j] : j;
    if (blk < 0 || blk >= q->hit_src_blocks)
        return NULL;
    return q->hit_src + blk * q->hit_block_stride + s * q->hit_token_stride
         + (int64_t)l * q->hit_layer_stride;
}

static const uint8_t *miss_row(const oracle_req *q, int32_t l, int64_t t_miss_idx)
{
    return q->miss_src + t_miss_idx * q->miss_token_stride + (int64_t)l * q->miss_layer_stride;
}

static uint8_t *pool_slot(const oracle_geom *g, uint8_t *pool, int32_t l, int32_t p,
                          int64_t b, int64_t s)
{
    return pool + ((((int64_t)l * g->P + p) * g->n_pool + b) * g->B + s) * g->Rp;
}

static int note(int *status, int code) { if (code > *status) *status = code; return code; }

/* ---- plan ------------------------------------------------------------------ */

/* Exclusive prefix sums over requests and the (request, block) work list.
 * Work item i = blk_off[r] + j is logical block j of request r.
 * Status: EINVAL for a negative count (detail = request); ERANGE when sum(nblk)
 * exceeds `capacity` (detail = sum), or when item i's pool block id is outside
 * [0, n_pool) or, for j < ceil(T_hit/B), its full block id is outside
 * [0, hit_src_blocks) (detail = smallest such i); EDUP, when check_injective, if a
 * pool block id is used twice (detail = smallest such id).  The larger code wins
 * when several apply. */
int oracle_plan(int32_t n_req, const oracle_req *reqs, int32_t B, const int32_t *tables,
                int64_t n_pool, int32_t check_injective, int64_t capacity,
                int64_t *tok_off, int64_t *hit_off, int64_t *blk_off,
                int32_t *item_req, int32_t *item_blk, int64_t *n_items, int64_t *detail)
{
    int status = OR_OK;
    int64_t det[8];
    for (int k = 0; k < 8; k++) det[k] = INT64_MAX;
    if (n_req < 0 || B <= 0 || n_pool <= 0) { *detail = -1; *n_items = 0; return OR_EINVAL; }

    tok_off[0] = hit_off[0] = blk_off[0] = 0;
    for (int32_t r = 0; r < n_req; r++) {
        const oracle_req *q = &reqs[r];
        if (q->t_hit < 0 || q->t_miss < 0) {
            note(&status, OR_EINVAL);
            if (r < det[OR_EINVAL]) det[OR_EINVAL] = r;
        }
        int64_t th = q->t_hit > 0 ? q->t_hit : 0, tm = q->t_miss > 0 ? q->t_miss : 0;
        tok_off[r + 1] = tok_off[r] + th + tm;
        hit_off[r + 1] = hit_off[r] + th;
        blk_off[r + 1] = blk_off[r] + ceil_div(th + tm, B);
    }
    *n_items = blk_off[n_req];
    if (status != OR_OK) { *detail = det[status]; return status; }
    if (*n_items > capacity) { *detail = *n_items; return OR_ERANGE; }

    for (int32_t r = 0; r < n_req; r++)
        for (int64_t j = 0; j < blk_off[r + 1] - blk_off[r]; j++) {
            item_req[blk_off[r] + j] = r;
            item_blk[blk_off[r] + j] = (int32_t)j;
        }

    uint8_t *seen = check_injective ? (uint8_t *)calloc((size_t)n_pool, 1) : NULL;
    for (int64_t i = 0; i < *n_items; i++) {
        const oracle_req *q = &reqs[item_req[i]];
        int64_t j = item_blk[i];
        int bad = 0;
        if (j < ceil_div(q->t_hit, B)) {
            int64_t sb = q->hit_src_table ? q->hit_src_table[j] : j;
            if (sb < 0 || sb >= q->hit_src_blocks) bad = 1;
        }
        int64_t b = tables[i];
        if (b < 0 || b >= n_pool) bad = 1;
        if (bad) {
            note(&status, OR_ERANGE);
            if (i < det[OR_ERANGE]) det[OR_ERANGE] = i;
            continue;
        }
        if (seen) {
            if (seen[b]) {
                note(&status, OR_EDUP);
                if (b < det[OR_EDUP]) det[OR_EDUP] = b;
            }
            seen[b] = 1;
        }
    }
    free(seen);
    *detail = status == OR_OK ? 0 : det[status];
    return status;
}

/* ---- the steps ------------------------------------------------------------- */

/* slice_layer: hit rows of layer l, requests packed in order ([sum T_hit][P][Rp]). */
int oracle_slice_layer(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                       int32_t layer, uint8_t *hit_out)
{
    int status = OR_OK;
    const int64_t R = (int64_t)g->P * g->Rp;
    int64_t row0 = 0;
    for (int32_t r = 0; r < n_req; r++) {
        const oracle_req *q = &reqs[r];
        for (int64_t t = 0; t < q->t_hit; t++) {
            const uint8_t *src = hit_row(g, q, layer, t);
            if (!src) { note(&status, OR_ERANGE); continue; }
            memcpy(hit_out + (row0 + t) * R, src, (size_t)R);
        }
        row0 += q->t_hit;
    }
    return status;
}

/* concatenate_tokens: complete_layer = hit_layer rows then miss_layer rows, for
 * every request, packed in order ([sum T_all][P][Rp]).  hit_layer is the output
 * of oracle_slice_layer for the same layer. */
int oracle_concatenate_tokens(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                              int32_t layer, const uint8_t *hit_layer, uint8_t *complete_out)
{
    const int64_t R = (int64_t)g->P * g->Rp;
    int64_t hit0 = 0, row0 = 0;
    for (int32_t r = 0; r < n_req; r++) {
        const oracle_req *q = &reqs[r];
        for (int64_t t = 0; t < q->t_hit; t++)
            memcpy(complete_out + (row0 + t) * R, hit_layer + (hit0 + t) * R, (size_t)R);
        for (int64_t m = 0; m < q->t_miss; m++)
            memcpy(complete_out + (row0 + q->t_hit + m) * R, miss_row(q, layer, m), (size_t)R);
        hit0 += q->t_hit;
        row0 += t_all_of(q);
    }
    return OR_OK;
}

/* Scatter complete_layer into the paged pool through each request's block table. */
int oracle_scatter_paged(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                         const int32_t *tables, int32_t layer, const uint8_t *complete_layer,
                         uint8_t *pool)
{
    int status = OR_OK;
    const int64_t R = (int64_t)g->P * g->Rp;
    int64_t row0 = 0, tab0 = 0;
    for (int32_t r = 0; r < n_req; r++) {
        const oracle_req *q = &reqs[r];
        int64_t ta = t_all_of(q);
        for (int64_t t = 0; t < ta; t++) {
            int64_t b = tables[tab0 + t / g->B];
            if (b < 0 || b >= g->n_pool) { note(&status, OR_ERANGE); continue; }
            for (int32_t p = 0; p < g->P; p++)
                memcpy(pool_slot(g, pool, layer, p, b, t % g->B),
                       complete_layer + (row0 + t) * R + (int64_t)p * g->Rp, (size_t)g->Rp);
        }
        row0 += ta;
        tab0 += ceil_div(ta, g->B);
    }
    return status;
}

/* The merge-scatter of one layer, composed from the three steps above in order:
 * slice_layer, concatenate_tokens, scatter into the pool.  complete_out, if not
 * NULL, receives complete_layer. */
int oracle_merge_scatter(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                         const int32_t *tables, int32_t layer, uint8_t *pool,
                         uint8_t *complete_out)
{
    const int64_t R = (int64_t)g->P * g->Rp;
    int64_t n_hit = 0, n_all = 0;
    for (int32_t r = 0; r < n_req; r++) { n_hit += reqs[r].t_hit; n_all += t_all_of(&reqs[r]); }
    uint8_t *hit_layer = (uint8_t *)malloc((size_t)(n_hit * R + 1));
    uint8_t *complete = complete_out ? complete_out : (uint8_t *)malloc((size_t)(n_all * R + 1));
    if (!hit_layer || !complete) { free(hit_layer); if (!complete_out) free(complete); return OR_EINVAL; }
    int status = oracle_slice_layer(g, n_req, reqs, layer, hit_layer);
    oracle_concatenate_tokens(g, n_req, reqs, layer, hit_layer, complete);
    int s2 = oracle_scatter_paged(g, n_req, reqs, tables, layer, complete, pool);
    if (s2 > status) status = s2;
    free(hit_layer);
    if (!complete_out) free(complete);
    return status;
}

/* Gather layer l's paged blocks into each request's contiguous K/V objects. */
int oracle_gather_objects(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                          const int32_t *tables, int32_t layer, const uint8_t *pool)
{
    int status = OR_OK;
    const int64_t obj_bytes = (int64_t)g->B * g->Rp;
    int64_t tab0 = 0;
    for (int32_t r = 0; r < n_req; r++) {
        const oracle_req *q = &reqs[r];
        int64_t nblk = ceil_div(t_all_of(q), g->B);
        for (int32_t p = 0; p < g->P; p++)
            for (int64_t j = 0; j < nblk; j++) {
                int64_t b = tables[tab0 + j];
                if (b < 0 || b >= g->n_pool) { note(&status, OR_ERANGE); continue; }
                uint8_t *obj = q->objects + (int64_t)layer * q->obj_layer_stride
                             + (int64_t)p * q->obj_plane_stride + j * q->obj_block_stride;
                memcpy(obj, pool_slot(g, (uint8_t *)pool, layer, p, b, 0), (size_t)obj_bytes);
            }
        tab0 += nblk;
    }
    return status;
}

/* Scatter each request's layer-l K/V objects back into its paged blocks. */
int oracle_scatter_back(const oracle_geom *g, int32_t n_req, const oracle_req *reqs,
                        const int32_t *tables, int32_t layer, uint8_t *pool)
{
    int status = OR_OK;
    const int64_t obj_bytes = (int64_t)g->B * g->Rp;
    int64_t tab0 = 0;
    for (int32_t r = 0; r < n_req; r++) {
        const oracle_req *q = &reqs[r];
        int64_t nblk = ceil_div(t_all_of(q), g->B);
        for (int32_t p = 0; p < g->P; p++)
            for (int64_t j = 0; j < nblk; j++) {
                int64_t b = tables[tab0 + j];
                if (b < 0 || b >= g->n_pool) { note(&status, OR_ERANGE); continue; }
                const uint8_t *obj = q->objects + (int64_t)layer * q->obj_layer_stride
                                   + (int64_t)p * q->obj_plane_stride + j * q->obj_block_stride;
                memcpy(pool_slot(g, pool, layer, p, b, 0), obj, (size_t)obj_bytes);
            }
        tab0 += nblk;
    }
    return status;
}

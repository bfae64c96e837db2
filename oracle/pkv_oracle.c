/*
 * Paged-KV attention oracle -- TEST INFRASTRUCTURE, not part of the library.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this file's shared object. The CUDA library never calls it, and the two
 * share no code, header or constant.
 *
 * It is the plain, slow, obviously correct statement of one model step of
 * paged-KV attention, in double precision, following:
 *
 *   Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five
 *   clients, up to 1.97x llama.cpp":
 *     - §Paged KV and paged attention: KV lives in fixed-size physical blocks
 *       of a shared pool; each sequence's block table maps logical token
 *       positions to physical blocks; attention reads the cached history by
 *       visiting that sequence's blocks in logical token order.
 *     - §Chunked prefill is a slot phase: each selected chunk appends directly
 *       to its slot's paged KV.
 *     - §Packing unequal prompt chunks together: several prompt chunks and
 *       decode rows share one token axis; per-query causal positions let them
 *       coexist in the same attention call.
 *   mlxcel manual, "Continuous batching", §Paged KV cache and prefix sharing:
 *     the block-table kernel and the gather path compute the same attention.
 *
 * The pages do not write the attention formula; the readings taken here are
 * ordinary causal grouped-query softmax attention:
 *   - query row i of a segment with n new rows and context length L sits at
 *     position p = L - n + i and sees keys 0..p (diagonal included);
 *   - q head h reads kv head floor(h / G), G = Hq / Hkv;
 *   - scores are scale * <q, k>, softmax over the visible keys.
 * Inputs are bfloat16 bit patterns, widened exactly; all arithmetic is double.
 *
 * Layouts (row-major, contiguous):
 *   pool      [num_blocks][Hkv][block_size][D]
 *   q         [T][Hq][D]              (packed rows)
 *   out       [T][Hq][D]              (double)
 *   block_tables [max_slots][max_blocks_per_slot]
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_SLOT (-1)
#define ORACLE_BAD_POSITION (-2)
#define ORACLE_BAD_BLOCK (-3)
#define ORACLE_BAD_SHAPE (-4)
#define ORACLE_NO_MEMORY (-5)

static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Physical pool row of each token: the token at logical position p of the
 * sequence in slot s lives in block block_tables[s][p / block_size], at row
 * p % block_size of that block (§Paged KV and paged attention).
 */
int oracle_slot_mapping(const int32_t *block_tables, int32_t max_slots,
                        int32_t max_blocks_per_slot, int32_t block_size,
                        int64_t num_blocks, const int32_t *token_slot,
                        const int32_t *token_pos, int64_t num_tokens,
                        int64_t *slot_mapping)
{
    for (int64_t t = 0; t < num_tokens; ++t) {
        int32_t s = token_slot[t];
        int32_t p = token_pos[t];
        if (s < 0 || s >= max_slots)
            return ORACLE_BAD_SLOT;
        if (p < 0 || p / block_size >= max_blocks_per_slot)
            return ORACLE_BAD_POSITION;
        int32_t block = block_tables[(int64_t)s * max_blocks_per_slot + p / block_size];
        if (block < 0 || block >= num_blocks)
            return ORACLE_BAD_BLOCK;
        slot_mapping[t] = (int64_t)block * block_size + p % block_size;
    }
    return ORACLE_OK;
}

/*
 * Append new tokens' keys and values to the pool: a plain copy of bit
 * patterns to the row named by slot_mapping (negative entries are skipped).
 */
int oracle_cache_write(const uint16_t *k_new, const uint16_t *v_new,
                       const int64_t *slot_mapping, int64_t num_tokens,
                       uint16_t *k_pool, uint16_t *v_pool, int64_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim)
{
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= num_blocks * block_size)
            return ORACLE_BAD_BLOCK;
        int64_t block = s / block_size;
        int64_t row = s % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            int64_t dst = ((block * num_kv_heads + h) * block_size + row) * head_dim;
            int64_t src = (t * num_kv_heads + h) * head_dim;
            memcpy(k_pool + dst, k_new + src, (size_t)head_dim * sizeof(uint16_t));
            memcpy(v_pool + dst, v_new + src, (size_t)head_dim * sizeof(uint16_t));
        }
    }
    return ORACLE_OK;
}

/* Softmax attention of one query vector over keys/values 0..p, in double. */
typedef const uint16_t *(*row_fn)(const void *ctx, int32_t j);

static void attend_row(const uint16_t *qv, int32_t p, int32_t head_dim, double scale,
                       row_fn key_row, row_fn value_row, const void *ctx,
                       double *scores, double *o)
{
    double m = -INFINITY;
    for (int32_t j = 0; j <= p; ++j) {
        const uint16_t *kj = key_row(ctx, j);
        double dot = 0.0;
        for (int32_t d = 0; d < head_dim; ++d)
            dot += widen_bf16(qv[d]) * widen_bf16(kj[d]);
        scores[j] = scale * dot;
        if (scores[j] > m)
            m = scores[j];
    }
    double denom = 0.0;
    for (int32_t d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    for (int32_t j = 0; j <= p; ++j) {
        double w = exp(scores[j] - m);
        const uint16_t *vj = value_row(ctx, j);
        denom += w;
        for (int32_t d = 0; d < head_dim; ++d)
            o[d] += w * widen_bf16(vj[d]);
    }
    for (int32_t d = 0; d < head_dim; ++d)
        o[d] /= denom;
}

/* ---- paged form: keys reached through the block table ---------------- */

typedef struct {
    const uint16_t *k_pool, *v_pool;
    const int32_t *table; /* this slot's block-table row */
    int32_t block_size, num_kv_heads, head_dim, kv_head;
} paged_ctx;

static const uint16_t *paged_row(const uint16_t *pool, const paged_ctx *c, int32_t j)
{
    int64_t block = c->table[j / c->block_size];
    int64_t row = j % c->block_size;
    return pool + ((block * c->num_kv_heads + c->kv_head) * c->block_size + row) * c->head_dim;
}

static const uint16_t *paged_key(const void *ctx, int32_t j)
{
    const paged_ctx *c = (const paged_ctx *)ctx;
    return paged_row(c->k_pool, c, j);
}

static const uint16_t *paged_value(const void *ctx, int32_t j)
{
    const paged_ctx *c = (const paged_ctx *)ctx;
    return paged_row(c->v_pool, c, j);
}

typedef struct {
    const uint16_t *q;
    const int32_t *cu_seqlens_q, *seq_slot, *context_lens, *block_tables;
    int32_t num_seqs, max_slots, max_blocks_per_slot, block_size;
    const uint16_t *k_pool, *v_pool;
    int64_t num_blocks;
    int32_t num_q_heads, num_kv_heads, head_dim;
    double scale;
    const uint8_t *row_mask; /* NULL = every row */
    double *out;
    int64_t next_task; /* (segment, kv head) work counter */
    int status;
} paged_job;

static int check_segment(const paged_job *J, int32_t s)
{
    int32_t slot = J->seq_slot[s];
    if (slot < 0 || slot >= J->max_slots)
        return ORACLE_BAD_SLOT;
    int32_t n = J->cu_seqlens_q[s + 1] - J->cu_seqlens_q[s];
    int32_t L = J->context_lens[slot];
    if (n < 0 || n > L || L > J->max_blocks_per_slot * J->block_size)
        return ORACLE_BAD_SHAPE;
    const int32_t *table = J->block_tables + (int64_t)slot * J->max_blocks_per_slot;
    for (int32_t b = 0; b < (L + J->block_size - 1) / J->block_size; ++b)
        if (n > 0 && (table[b] < 0 || table[b] >= J->num_blocks))
            return ORACLE_BAD_BLOCK;
    return ORACLE_OK;
}

static void paged_task(paged_job *J, int32_t s, int32_t g, double *scores)
{
    int32_t slot = J->seq_slot[s];
    int32_t n = J->cu_seqlens_q[s + 1] - J->cu_seqlens_q[s];
    int32_t L = J->context_lens[slot];
    int32_t G = J->num_q_heads / J->num_kv_heads;
    paged_ctx c = {J->k_pool, J->v_pool,
                   J->block_tables + (int64_t)slot * J->max_blocks_per_slot,
                   J->block_size, J->num_kv_heads, J->head_dim, g};
    for (int32_t i = 0; i < n; ++i) {
        int64_t row = J->cu_seqlens_q[s] + i;
        if (J->row_mask && !J->row_mask[row])
            continue;
        int32_t p = L - n + i;
        for (int32_t h = g * G; h < (g + 1) * G; ++h) {
            const uint16_t *qv = J->q + (row * J->num_q_heads + h) * J->head_dim;
            double *o = J->out + (row * J->num_q_heads + h) * J->head_dim;
            attend_row(qv, p, J->head_dim, J->scale, paged_key, paged_value, &c, scores, o);
        }
    }
}

static void *paged_worker(void *arg)
{
    paged_job *J = (paged_job *)arg;
    int64_t max_ctx = (int64_t)J->max_blocks_per_slot * J->block_size;
    double *scores = (double *)malloc((size_t)(max_ctx > 0 ? max_ctx : 1) * sizeof(double));
    if (!scores) {
        __atomic_store_n(&J->status, ORACLE_NO_MEMORY, __ATOMIC_SEQ_CST);
        return NULL;
    }
    int64_t tasks = (int64_t)J->num_seqs * J->num_kv_heads;
    for (;;) {
        int64_t t = __atomic_fetch_add(&J->next_task, 1, __ATOMIC_SEQ_CST);
        if (t >= tasks)
            break;
        paged_task(J, (int32_t)(t / J->num_kv_heads), (int32_t)(t % J->num_kv_heads), scores);
    }
    free(scores);
    return NULL;
}

static int run_threads(void *(*fn)(void *), void *job, int32_t num_threads)
{
    if (num_threads <= 1) {
        fn(job);
        return ORACLE_OK;
    }
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)num_threads);
    if (!tids)
        return ORACLE_NO_MEMORY;
    int32_t started = 0;
    for (; started < num_threads; ++started)
        if (pthread_create(&tids[started], NULL, fn, job) != 0)
            break;
    if (started == 0)
        fn(job);
    for (int32_t i = 0; i < started; ++i)
        pthread_join(tids[i], NULL);
    free(tids);
    return ORACLE_OK;
}

/*
 * Attention over the pool for every packed row (or the rows whose row_mask
 * byte is non-zero). Writes out[T][Hq][D] in double; rows left out of the
 * mask are not touched. Work is split over (segment, kv head) tasks.
 */
int oracle_attention_paged(const uint16_t *q, const int32_t *cu_seqlens_q, int32_t num_seqs,
                           const int32_t *seq_slot, const int32_t *context_lens,
                           const int32_t *block_tables, int32_t max_slots,
                           int32_t max_blocks_per_slot, int32_t block_size,
                           const uint16_t *k_pool, const uint16_t *v_pool, int64_t num_blocks,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           double scale, const uint8_t *row_mask, double *out,
                           int32_t num_threads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0)
        return ORACLE_BAD_SHAPE;
    paged_job J = {q, cu_seqlens_q, seq_slot, context_lens, block_tables, num_seqs, max_slots,
                   max_blocks_per_slot, block_size, k_pool, v_pool, num_blocks, num_q_heads,
                   num_kv_heads, head_dim, scale, row_mask, out, 0, ORACLE_OK};
    for (int32_t s = 0; s < num_seqs; ++s) {
        int rc = check_segment(&J, s);
        if (rc != ORACLE_OK)
            return rc;
    }
    int rc = run_threads(paged_worker, &J, num_threads);
    return rc != ORACLE_OK ? rc : J.status;
}

/* ---- contiguous form: one sequence's history as [L][Hkv][D] ----------- */

typedef struct {
    const uint16_t *k, *v;
    int32_t num_kv_heads, head_dim, kv_head;
} dense_ctx;

static const uint16_t *dense_key(const void *ctx, int32_t j)
{
    const dense_ctx *c = (const dense_ctx *)ctx;
    return c->k + ((int64_t)j * c->num_kv_heads + c->kv_head) * c->head_dim;
}

static const uint16_t *dense_value(const void *ctx, int32_t j)
{
    const dense_ctx *c = (const dense_ctx *)ctx;
    return c->v + ((int64_t)j * c->num_kv_heads + c->kv_head) * c->head_dim;
}

/*
 * Causal attention of the last n positions of one sequence over its own
 * contiguous history k/v [L][Hkv][D]; q is [n][Hq][D], out [n][Hq][D].
 * This is the "attention over a contiguous cache" that the paged form must
 * equal (the gather path of the mlxcel manual's paged-KV section).
 */
int oracle_attention_dense(const uint16_t *q, int32_t n, const uint16_t *k, const uint16_t *v,
                           int32_t L, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           double scale, double *out)
{
    if (n < 0 || n > L || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return ORACLE_BAD_SHAPE;
    double *scores = (double *)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    if (!scores)
        return ORACLE_NO_MEMORY;
    int32_t G = num_q_heads / num_kv_heads;
    for (int32_t i = 0; i < n; ++i) {
        int32_t p = L - n + i;
        for (int32_t h = 0; h < num_q_heads; ++h) {
            dense_ctx c = {k, v, num_kv_heads, head_dim, h / G};
            attend_row(q + ((int64_t)i * num_q_heads + h) * head_dim, p, head_dim, scale,
                       dense_key, dense_value, &c, scores,
                       out + ((int64_t)i * num_q_heads + h) * head_dim);
        }
    }
    free(scores);
    return ORACLE_OK;
}

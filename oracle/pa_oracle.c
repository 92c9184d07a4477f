/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header or constant with the
 * CUDA library and reads no paged pool for attention: it works on each
 * sequence's LOGICAL, contiguous K/V history.
 *
 * What it computes, and where the pages fix it:
 *
 *  - Attention itself is unchanged by paging: "PagedAttention: memetakan blok
 *    KV logis ke memori fisik tidak kontigu" (nalar.dev), opening section
 *    (the attention equation does not change) and section "Paging tidak
 *    mengompresi KV cache secara matematis" (no pruning, no quantisation, no
 *    sparse attention: exact full attention over every retained token).  The
 *    cached values are the same as without paging: "Apa itu PagedAttention?"
 *    (gininih.com), section "Batasan dan salah paham umum".  The equation is
 *    the ordinary scaled dot-product attention, read plainly:
 *        S_j = (q . k_j) * scale,  o = sum_j exp(S_j - max S) v_j / sum_j exp(S_j - max S)
 *    with scale = 1/sqrt(d) supplied by the caller.
 *  - A query token at absolute position t attends to positions 0..t of its
 *    own sequence (autoregressive: every new token attends to all previous
 *    ones and itself): "Melihat Lebih Dalam vLLM v0.7" (bicarait.com), section
 *    "Blueprint Arsitektur 1: Akar Masalah Fragmentasi KV Cache"; for a
 *    prefill chunk the same rule gives the causal mask j <= P + i, section
 *    "Blueprint Arsitektur 3: Chunked Prefill".  Decode is the case of one
 *    query at t = L - 1.
 *  - Grouped query heads: query head h reads KV head h / (Hq/Hkv).  The pages
 *    say nothing about GQA; this contiguous-group reading is the plain one.
 *  - Slot of logical token j: block_table[j / bs] * bs + j % bs, the logical
 *    block -> physical block translation of the block table ("PagedAttention:
 *    memetakan blok KV logis ...", section "Urutan logis dipisahkan dari
 *    penempatan fisik", worked mapping 0,1,2,3 -> 17,4,29,8).
 *  - reshape_and_cache: only the new token's K and V are computed and stored
 *    ("KV Cache dan PagedAttention: Apa Fungsinya ...", section "Apa itu KV
 *    Cache?"); the store is a plain byte scatter into the slot's place in the
 *    pool laid out [num_blocks][Hkv][bs][d].
 *  - copy_blocks: copy-on-write gives a diverging branch its own copy of a
 *    shared block ("Apa itu PagedAttention?", section "Cara kerja
 *    PagedAttention", item 3; nalar.dev, section "Sharing blok dapat
 *    menghindari duplikasi state KV"): a plain byte copy of both caches.
 *
 * Every loop below is the definition written out; the only concession to
 * speed is that independent (sequence, query head) items are spread over
 * pthreads.  No blocking, no fusion, no reordering of any sum.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Attention                                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    const double *q, *k, *v;
    double *out;
    const int64_t *q_start;  /* [S+1] first query row of each sequence      */
    const int64_t *q_pos0;   /* [S]   absolute position of its first query  */
    const int64_t *kv_start; /* [S]   first K/V row of each sequence         */
    const int64_t *kv_len;   /* [S]   number of K/V rows of each sequence    */
    int S, Hq, Hkv, d;
    double scale;
    int nthreads, tid;
    int status;
} attn_job;

/* One (sequence s, query head h) item: every query row of s, head h. */
static int attend_one(const attn_job *J, int s, int h, double *scores)
{
    const int d = J->d;
    const int group = J->Hq / J->Hkv;
    const int hk = h / group; /* query head h reads KV head h / group */
    for (int64_t i = J->q_start[s]; i < J->q_start[s + 1]; ++i) {
        const int64_t t = J->q_pos0[s] + (i - J->q_start[s]); /* absolute position */
        if (t < 0 || t >= J->kv_len[s]) return 1;
        const double *qi = J->q + (i * J->Hq + h) * d;
        /* scores over positions 0..t (the query's own position included) */
        double mx = -INFINITY;
        for (int64_t j = 0; j <= t; ++j) {
            const double *kj = J->k + ((J->kv_start[s] + j) * J->Hkv + hk) * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += qi[c] * kj[c];
            scores[j] = dot * J->scale;
            if (scores[j] > mx) mx = scores[j];
        }
        double denom = 0.0;
        for (int64_t j = 0; j <= t; ++j) {
            scores[j] = exp(scores[j] - mx);
            denom += scores[j];
        }
        double *oi = J->out + (i * J->Hq + h) * d;
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        for (int64_t j = 0; j <= t; ++j) {
            const double *vj = J->v + ((J->kv_start[s] + j) * J->Hkv + hk) * d;
            const double w = scores[j] / denom;
            for (int c = 0; c < d; ++c) oi[c] += w * vj[c];
        }
    }
    return 0;
}

static void *attn_worker(void *arg)
{
    attn_job *J = (attn_job *)arg;
    int64_t max_len = 1;
    for (int s = 0; s < J->S; ++s)
        if (J->kv_len[s] > max_len) max_len = J->kv_len[s];
    double *scores = (double *)malloc(sizeof(double) * (size_t)max_len);
    if (!scores) { J->status = 2; return NULL; }
    int64_t item = 0;
    for (int s = 0; s < J->S; ++s)
        for (int h = 0; h < J->Hq; ++h, ++item)
            if (item % J->nthreads == J->tid && attend_one(J, s, h, scores)) J->status = 1;
    free(scores);
    return NULL;
}

/*
 * oracle_attention: causal attention of every query row over its sequence's
 * logical K/V.
 *   q   [n_q][Hq][d]   (n_q = q_start[S])
 *   k,v [n_kv][Hkv][d] (sequence s owns rows kv_start[s] .. kv_start[s]+kv_len[s]-1)
 *   out [n_q][Hq][d]
 * Returns 0, or 1 if a query position lies outside its sequence, or 2 on
 * allocation failure, or 3 on bad shapes.
 */
int oracle_attention(const double *q, const double *k, const double *v, double *out,
                     const int64_t *q_start, const int64_t *q_pos0,
                     const int64_t *kv_start, const int64_t *kv_len,
                     int S, int Hq, int Hkv, int d, double scale, int nthreads)
{
    if (S < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return 3;
    if (nthreads < 1) nthreads = 1;
    attn_job *jobs = (attn_job *)calloc((size_t)nthreads, sizeof(attn_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 2; }
    for (int t = 0; t < nthreads; ++t) {
        attn_job J = {q, k, v, out, q_start, q_pos0, kv_start, kv_len,
                      S, Hq, Hkv, d, scale, nthreads, t, 0};
        jobs[t] = J;
    }
    int rc = 0;
    if (nthreads == 1) {
        attn_worker(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, attn_worker, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    for (int t = 0; t < nthreads; ++t) if (jobs[t].status) rc = jobs[t].status;
    free(jobs);
    free(th);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Block table, slots and the byte-level cache operations                    */
/* ------------------------------------------------------------------------ */

/* slot of each logical token j in [0, n): table[j / bs] * bs + j % bs */
void oracle_slot_mapping(const int32_t *table, int64_t n, int bs, int64_t *slots)
{
    for (int64_t j = 0; j < n; ++j)
        slots[j] = (int64_t)table[j / bs] * bs + j % bs;
}

/*
 * oracle_reshape_and_cache: for each new token t with slot >= 0, copy its
 * K row and V row of every KV head into the pool place of that slot.
 *   k_new, v_new  [T][Hkv][d] elements of esize bytes
 *   k_cache, v_cache [num_blocks][Hkv][bs][d]
 * A negative slot is padding and is skipped.  Returns 1 if a slot is out of
 * the pool.
 */
int oracle_reshape_and_cache(const uint8_t *k_new, const uint8_t *v_new,
                             uint8_t *k_cache, uint8_t *v_cache,
                             const int64_t *slot_mapping, int64_t T,
                             int64_t num_blocks, int Hkv, int bs, int d, int esize)
{
    const size_t row = (size_t)d * (size_t)esize;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        const int64_t blk = slot / bs, off = slot % bs;
        if (blk >= num_blocks) return 1;
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (size_t)(((blk * Hkv + h) * bs + off)) * row;
            const size_t src = (size_t)(t * Hkv + h) * row;
            memcpy(k_cache + dst, k_new + src, row);
            memcpy(v_cache + dst, v_new + src, row);
        }
    }
    return 0;
}

/*
 * oracle_copy_blocks: for every (src, dst) pair, physical block dst of both
 * caches becomes a byte copy of block src.  Pairs are applied in order.
 */
int oracle_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, const int64_t *pairs, int64_t n,
                       int64_t num_blocks, int Hkv, int bs, int d, int esize)
{
    const size_t blk = (size_t)Hkv * (size_t)bs * (size_t)d * (size_t)esize;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) return 1;
        memmove(k_cache + (size_t)dst * blk, k_cache + (size_t)src * blk, blk);
        memmove(v_cache + (size_t)dst * blk, v_cache + (size_t)src * blk, blk);
    }
    return 0;
}

/*
 * pka_oracle.c -- float64 CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the test suite, the
 * package's smoke check and the benchmark's CPU-baseline leg may load or call
 * this code. It shares nothing with the CUDA library: no headers, no helpers,
 * no constants.
 *
 * What it computes is the plain definition the method reduces to. The ROCm
 * attention-backend pages ("Beyond porting", section "Three-path processing
 * explained") split one step into a cache write, a decode path, a varlen
 * prefill path and an extend path whose context chunks are combined by an LSE
 * merge; every one of those pieces computes, for a query at absolute position
 * p of request r and query head h,
 *
 *     s_j  = scale * <q, K[r, j, h / G]>        for keys j = 0 .. p
 *     lse  = log( sum_j exp(s_j) )              (natural log, scale included)
 *     o    = sum_j exp(s_j - lse) * V[r, j, h / G]
 *
 * with G = Hq / Hkv query heads per KV head, and K/V read by walking the
 * block table: block = block_table[r][j / bs], offset = j % bs.
 *
 * Layouts (caller's arrays, bf16 carried as uint16 bit patterns):
 *   q        [T, Hq, d]
 *   k_cache  [num_blocks, Hkv, bs, d]
 *   v_cache  [num_blocks, Hkv, bs, dv], or NULL for the MLA latent cache,
 *            where V is the first dv entries of the K row (page 1,
 *            "The hybrid processing strategy": decode works on the 576-dim
 *            latent; the value is its first 512 dims).
 *   block_table [B, max_blocks] int32, query_start_loc [B+1], seq_lens [B].
 * A request's new tokens are its last q_r = qsl[r+1]-qsl[r] positions, so
 * token i of request r sits at position p = seq_lens[r] - q_r + i.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_BLOCK 1
#define ORACLE_BAD_ARG 2
#define ORACLE_NO_MEMORY 3

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* reshape_and_cache: scatter new K/V rows into their slots (page 2, the      */
/* unified backend's stage 1 "save key/value into the KV cache").             */
/* slot < 0 means "do not write" (padding tokens).                            */
/* ------------------------------------------------------------------------ */
int oracle_cache_write(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                       int64_t num_tokens, int num_kv_heads, int head_dim, int head_dim_v,
                       uint16_t *k_cache, uint16_t *v_cache, int64_t num_blocks, int block_size)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        if (blk >= num_blocks)
            return ORACLE_BAD_BLOCK;
        for (int h = 0; h < num_kv_heads; ++h) {
            const uint16_t *src = k + ((size_t)t * num_kv_heads + h) * head_dim;
            uint16_t *dst = k_cache + (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim;
            memcpy(dst, src, (size_t)head_dim * sizeof(uint16_t));
            if (v && v_cache) {
                const uint16_t *vs = v + ((size_t)t * num_kv_heads + h) * head_dim_v;
                uint16_t *vd = v_cache + (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim_v;
                memcpy(vd, vs, (size_t)head_dim_v * sizeof(uint16_t));
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Attention over a key range, one (token, head) row at a time.               */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *block_table;
    int max_blocks;
    const int32_t *qsl, *seq_lens;
    int num_reqs;
    const int32_t *key_begin, *key_end; /* per request; NULL = [0, +inf) */
    int num_q_heads, num_kv_heads, head_dim, head_dim_v, block_size;
    int64_t num_blocks;
    double scale;
    const int64_t *rows; /* flattened t * Hq + h; NULL = all T * Hq rows */
    int64_t n_rows;
    double *out, *lse;
    int64_t row_begin, row_end;
    int status;
} attn_job;

static int find_request(const int32_t *qsl, int num_reqs, int64_t t)
{
    int lo = 0, hi = num_reqs - 1;
    while (lo < hi) { /* last r with qsl[r] <= t */
        int mid = (lo + hi + 1) / 2;
        if (qsl[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

static void *attn_worker(void *arg)
{
    attn_job *J = (attn_job *)arg;
    const int G = J->num_q_heads / J->num_kv_heads;
    const int d = J->head_dim, dv = J->head_dim_v, bs = J->block_size;
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);
    double *acc = (double *)malloc(sizeof(double) * (size_t)dv);
    double *scores = NULL;
    int64_t cap = 0;
    if (!qd || !acc) {
        J->status = ORACLE_NO_MEMORY;
        goto done;
    }
    for (int64_t i = J->row_begin; i < J->row_end; ++i) {
        int64_t flat = J->rows ? J->rows[i] : i;
        int64_t t = flat / J->num_q_heads;
        int h = (int)(flat % J->num_q_heads);
        int r = find_request(J->qsl, J->num_reqs, t);
        int64_t q_len = J->qsl[r + 1] - J->qsl[r];
        int64_t ctx = (int64_t)J->seq_lens[r] - q_len;
        int64_t p = ctx + (t - J->qsl[r]); /* absolute position of this query */
        int64_t j0 = 0, j1 = p + 1;        /* causal: keys 0 .. p */
        if (J->key_begin && J->key_begin[r] > j0)
            j0 = J->key_begin[r];
        if (J->key_end && J->key_end[r] < j1)
            j1 = J->key_end[r];
        int g = h / G; /* GQA: query head h reads kv head h / G */
        const uint16_t *qrow = J->q + ((size_t)t * J->num_q_heads + h) * d;
        for (int x = 0; x < d; ++x)
            qd[x] = bf16_to_double(qrow[x]);
        double *o = J->out + (size_t)i * dv;
        int64_t n = j1 > j0 ? j1 - j0 : 0;
        if (n == 0) { /* empty key set: o = 0, lse = -inf */
            for (int x = 0; x < dv; ++x)
                o[x] = 0.0;
            J->lse[i] = -INFINITY;
            continue;
        }
        if (n > cap) {
            free(scores);
            cap = n;
            scores = (double *)malloc(sizeof(double) * (size_t)cap);
            if (!scores) {
                J->status = ORACLE_NO_MEMORY;
                goto done;
            }
        }
        /* scores s_j = scale * q . k_j */
        double m = -INFINITY;
        for (int64_t j = j0; j < j1; ++j) {
            int64_t blk = J->block_table[(size_t)r * J->max_blocks + j / bs];
            if (blk < 0 || blk >= J->num_blocks) {
                J->status = ORACLE_BAD_BLOCK;
                goto done;
            }
            const uint16_t *krow = J->k_cache + (((size_t)blk * J->num_kv_heads + g) * bs + j % bs) * d;
            double s = 0.0;
            for (int x = 0; x < d; ++x)
                s += qd[x] * bf16_to_double(krow[x]);
            s *= J->scale;
            scores[j - j0] = s;
            if (s > m)
                m = s;
        }
        /* softmax-weighted sum of V, normalised by l = sum exp(s - m) */
        double l = 0.0;
        for (int x = 0; x < dv; ++x)
            acc[x] = 0.0;
        for (int64_t j = j0; j < j1; ++j) {
            double w = exp(scores[j - j0] - m);
            l += w;
            int64_t blk = J->block_table[(size_t)r * J->max_blocks + j / bs];
            const uint16_t *vrow = J->v_cache
                ? J->v_cache + (((size_t)blk * J->num_kv_heads + g) * bs + j % bs) * dv
                : J->k_cache + (((size_t)blk * J->num_kv_heads + g) * bs + j % bs) * d;
            for (int x = 0; x < dv; ++x)
                acc[x] += w * bf16_to_double(vrow[x]);
        }
        for (int x = 0; x < dv; ++x)
            o[x] = acc[x] / l;
        J->lse[i] = m + log(l);
    }
done:
    free(qd);
    free(acc);
    free(scores);
    return NULL;
}

/*
 * oracle_attention: out[i, :dv] and lse[i] for each requested row i
 * (rows[i] = t * Hq + h, or every row in order when rows == NULL).
 * key_begin / key_end (per request, may be NULL) restrict the keys to
 * [key_begin[r], key_end[r]) on top of the causal bound j <= p; with both NULL
 * this is full attention. Runs on `nthreads` POSIX threads (<= 0 means 1).
 */
int oracle_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                     const int32_t *block_table, int max_blocks, const int32_t *query_start_loc,
                     const int32_t *seq_lens, int num_reqs, const int32_t *key_begin,
                     const int32_t *key_end, int num_q_heads, int num_kv_heads, int head_dim,
                     int head_dim_v, int block_size, int64_t num_blocks, double scale,
                     const int64_t *rows, int64_t n_rows, double *out, double *lse, int nthreads)
{
    if (num_reqs <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0 ||
        head_dim <= 0 || head_dim_v <= 0 || (!v_cache && head_dim_v > head_dim))
        return ORACLE_BAD_ARG;
    if (!rows)
        n_rows = (int64_t)query_start_loc[num_reqs] * num_q_heads;
    if (nthreads <= 0)
        nthreads = 1;
    if (nthreads > n_rows)
        nthreads = n_rows > 0 ? (int)n_rows : 1;
    attn_job *jobs = (attn_job *)calloc((size_t)nthreads, sizeof(attn_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return ORACLE_NO_MEMORY;
    }
    for (int w = 0; w < nthreads; ++w) {
        attn_job *J = &jobs[w];
        J->q = q;
        J->k_cache = k_cache;
        J->v_cache = v_cache;
        J->block_table = block_table;
        J->max_blocks = max_blocks;
        J->qsl = query_start_loc;
        J->seq_lens = seq_lens;
        J->num_reqs = num_reqs;
        J->key_begin = key_begin;
        J->key_end = key_end;
        J->num_q_heads = num_q_heads;
        J->num_kv_heads = num_kv_heads;
        J->head_dim = head_dim;
        J->head_dim_v = head_dim_v;
        J->block_size = block_size;
        J->num_blocks = num_blocks;
        J->scale = scale;
        J->rows = rows;
        J->n_rows = n_rows;
        J->out = out;
        J->lse = lse;
        J->row_begin = n_rows * w / nthreads;
        J->row_end = n_rows * (w + 1) / nthreads;
        J->status = ORACLE_OK;
    }
    int spawned = 0;
    for (int w = 1; w < nthreads; ++w)
        if (pthread_create(&tid[w], NULL, attn_worker, &jobs[w]) == 0)
            spawned = w;
        else
            break;
    /* rows of workers that could not be started run on this thread */
    for (int w = spawned + 1; w < nthreads; ++w)
        attn_worker(&jobs[w]);
    attn_worker(&jobs[0]);
    for (int w = 1; w <= spawned; ++w)
        pthread_join(tid[w], NULL);
    int status = ORACLE_OK;
    for (int w = 0; w < nthreads; ++w)
        if (jobs[w].status != ORACLE_OK)
            status = jobs[w].status;
    free(jobs);
    free(tid);
    return status;
}

/*
 * merge_attn_states (page 2, extend path: "each chunk yields an output and an
 * LSE ... the LSE captures the softmax denominator, allowing a numerically
 * stable merge"). Two partial results over disjoint key sets combine as
 *     m = max(la, lb), wa = exp(la - m), wb = exp(lb - m)
 *     o = (wa * oa + wb * ob) / (wa + wb),  lse = m + log(wa + wb).
 * A side with lse = -inf (no keys) contributes nothing; both empty gives
 * o = 0, lse = -inf.
 */
void oracle_merge_attn_states(int64_t n_rows, int head_dim_v, const double *a_out, const double *a_lse,
                              const double *b_out, const double *b_lse, double *out, double *out_lse)
{
    for (int64_t i = 0; i < n_rows; ++i) {
        double la = a_lse[i], lb = b_lse[i];
        double *o = out + (size_t)i * head_dim_v;
        const double *oa = a_out + (size_t)i * head_dim_v;
        const double *ob = b_out + (size_t)i * head_dim_v;
        if (la == -INFINITY && lb == -INFINITY) {
            for (int x = 0; x < head_dim_v; ++x)
                o[x] = 0.0;
            out_lse[i] = -INFINITY;
            continue;
        }
        double m = la > lb ? la : lb;
        double wa = exp(la - m), wb = exp(lb - m);
        for (int x = 0; x < head_dim_v; ++x)
            o[x] = (wa * oa[x] + wb * ob[x]) / (wa + wb);
        out_lse[i] = m + log(wa + wb);
    }
}

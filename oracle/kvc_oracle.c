/*
 * kvc_oracle.c -- plain, slow CPU oracle for paged KV storage and paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this
 * file: only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
 * shares no code, header or constant with the CUDA library; the two meet only through
 * the seeded input generators.
 *
 * Floating point is fp64 throughout, except the INT8 quantiser, whose integer codes are
 * decided in fp32 (the precision the device decides them in; the pages fix none).  bf16
 * inputs are widened exactly (a bf16 value is the top 16 bits of an fp32 value) and never
 * rounded again.
 *
 * Sources (page title, section):
 *   [KV]   Quail "KV", sections "Paged KV", "KV rewind", "The sharing plan"
 *   [TI]   TileInfer.jl "KV cache", sections "Pages and block tables",
 *          "Growing, rolling back, releasing", "INT8 cache"
 *   [PA]   "KV Cache Management and PagedAttention", sections "Connect token order to
 *          storage locations", "Grow the allocation as generation proceeds",
 *          "Compute attention over scattered KV"
 *
 * Conventions (the plain readings where the pages leave a step open):
 *   - positions, logical blocks, page ids and slots are 0-based ([PA] says both block
 *     indices and positions inside a block start at 0);
 *   - a pool is [num_pages][page_size][kv_heads][head_dim], so the vector of one
 *     (slot, kv head) is head_dim contiguous values at ((slot*kv_heads)+g)*head_dim;
 *   - q head h reads kv head h / (q_heads / kv_heads) (contiguous GQA groups);
 *   - context_lens[s] counts every position of sequence s including the new ones: the
 *     newest token's query also attends to that token's own key and value ([PA],
 *     "Compute attention over scattered KV", position 8 attends over 9 positions);
 *   - new token i of sequence s (0 <= i < q_len) sits at position ctx - q_len + i and sees
 *     keys 0 .. ctx - q_len + i (causal);
 *   - scores are scaled by `scale` (1/sqrt(head_dim) unless the caller says otherwise);
 *   - lse is the natural-log log-sum-exp of the scaled scores; a query with no visible key
 *     gets output 0 and lse = -inf.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Widen one bf16 bit pattern to fp64: the pattern is the high half of an IEEE fp32. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Address rule.  [TI] "Pages and block tables": position p lives in the page the block
 * table lists at index p / page_size, at offset p % page_size.  [PA] "Connect token
 * order to storage locations": position 6 with 4-slot blocks is logical block 1, slot 2.
 * The slot flattens (page, offset) into one index into the pool: page * page_size +
 * offset ([TI], same section).
 */
int64_t kvo_slot_of_position(const int32_t *block_table, int64_t bt_stride, int64_t seq,
                             int64_t position, int64_t page_size)
{
    int64_t logical_block = position / page_size;
    int64_t offset = position % page_size;
    int64_t page = block_table[seq * bt_stride + logical_block];
    return page * page_size + offset;
}

/*
 * Slots of every new token of every sequence.  [TI] "Pages and block tables": before a
 * step, each new token gets its slot.  Sequence s owns tokens q_indptr[s] ..
 * q_indptr[s+1]-1; token i of s is at position context_lens[s] - q_len + i.  A token with
 * no position (context_lens[s] < q_len) is padding and gets slot -1, which the store skips.
 */
void kvo_slot_mapping(const int32_t *block_table, int64_t bt_stride,
                      const int32_t *context_lens, const int32_t *q_indptr, int64_t num_seqs,
                      int64_t page_size, int64_t *slots_out)
{
    for (int64_t s = 0; s < num_seqs; ++s) {
        int64_t first = q_indptr[s];
        int64_t q_len = q_indptr[s + 1] - first;
        for (int64_t i = 0; i < q_len; ++i) {
            int64_t position = (int64_t)context_lens[s] - q_len + i;
            slots_out[first + i] =
                position < 0 ? -1
                             : kvo_slot_of_position(block_table, bt_stride, s, position,
                                                    page_size);
        }
    }
}

/*
 * Store.  [TI] "Pages and block tables": the new keys and values are written at their
 * slots.  A slot below zero marks a padding token and is skipped.  The copy is of bit
 * patterns, so NaN payloads and signed zeros travel unchanged.
 */
void kvo_store(uint16_t *k_pool, uint16_t *v_pool, int64_t kv_heads, int64_t head_dim,
               const uint16_t *k_new, const uint16_t *v_new, const int64_t *slots,
               int64_t num_tokens)
{
    int64_t row = kv_heads * head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        if (slots[t] < 0)
            continue;
        for (int64_t e = 0; e < row; ++e) {
            k_pool[slots[t] * row + e] = k_new[t * row + e];
            v_pool[slots[t] * row + e] = v_new[t * row + e];
        }
    }
}

/*
 * Copy-on-write page copy ([PA] "Split shared blocks when a write is needed": the shared
 * block is copied to a new block, keeping the KV already in it, before the writer's table
 * entry is pointed at the copy).  Every copy reads the pools as they were before the call:
 * the sources are copied aside first, then written to their destinations.
 */
void kvo_copy_pages(uint16_t *k_pool, uint16_t *v_pool, int64_t page_elems,
                    const int64_t *src_pages, const int64_t *dst_pages, int64_t num_copies,
                    uint16_t *scratch_k, uint16_t *scratch_v)
{
    for (int64_t i = 0; i < num_copies; ++i)
        for (int64_t e = 0; e < page_elems; ++e) {
            scratch_k[i * page_elems + e] = k_pool[src_pages[i] * page_elems + e];
            scratch_v[i * page_elems + e] = v_pool[src_pages[i] * page_elems + e];
        }
    for (int64_t i = 0; i < num_copies; ++i)
        for (int64_t e = 0; e < page_elems; ++e) {
            k_pool[dst_pages[i] * page_elems + e] = scratch_k[i * page_elems + e];
            v_pool[dst_pages[i] * page_elems + e] = scratch_v[i * page_elems + e];
        }
}

/*
 * INT8 quantisation of one (position, kv head) vector ([TI] "INT8 cache"): x ~ scale * code,
 * symmetric, scale = max |x| / 127, codes rounded to nearest (ties to even) and kept in
 * [-127, 127]; done once, when the position is written.  The pages fix no precision for the
 * scale, so it is computed in fp32 (max and quotient both fp32, rounded to nearest), the
 * precision the device takes the same integer decision in.  An all-zero vector gets scale 0
 * and codes 0.
 */
void kvo_quantize_vector(const uint16_t *x, int64_t n, int8_t *codes, float *scale)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf((float)bf16_bits_to_double(x[i]));
        if (a > m)
            m = a;
    }
    float sc = m / 127.0f;
    *scale = sc;
    for (int64_t i = 0; i < n; ++i) {
        if (sc == 0.0f) {
            codes[i] = 0;
            continue;
        }
        float r = rintf((float)bf16_bits_to_double(x[i]) / sc);
        if (r > 127.0f)
            r = 127.0f;
        if (r < -127.0f)
            r = -127.0f;
        codes[i] = (int8_t)r;
    }
}

/*
 * Store into INT8 pages: token t's K and V vectors of every kv head are quantised and
 * written at slot_mapping[t] (slot < 0: skipped).
 *   k_codes/v_codes [num_pages][page_size][kv_heads][head_dim] int8
 *   k_scales/v_scales [num_pages][kv_heads][page_size] fp32
 *   k_new/v_new [num_tokens][kv_heads][head_dim] bf16 bits
 */
void kvo_store_int8(int8_t *k_codes, int8_t *v_codes, float *k_scales, float *v_scales,
                    int64_t page_size, int64_t kv_heads, int64_t head_dim,
                    const uint16_t *k_new, const uint16_t *v_new, const int64_t *slots,
                    int64_t num_tokens)
{
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slots[t];
        if (slot < 0)
            continue;
        int64_t page = slot / page_size, off = slot % page_size;
        for (int64_t g = 0; g < kv_heads; ++g) {
            int64_t src = (t * kv_heads + g) * head_dim;
            int64_t dst = (slot * kv_heads + g) * head_dim;
            int64_t sidx = (page * kv_heads + g) * page_size + off;
            kvo_quantize_vector(k_new + src, head_dim, k_codes + dst, &k_scales[sidx]);
            kvo_quantize_vector(v_new + src, head_dim, v_codes + dst, &v_scales[sidx]);
        }
    }
}

/* ---------------------------------------------------------------------------------- */
/* Attention                                                                          */
/* ---------------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *q, *k_pool, *v_pool;
    int64_t page_size, kv_heads, head_dim, q_heads;
    const int32_t *block_table;
    int64_t bt_stride;
    const int32_t *context_lens, *q_indptr;
    int64_t num_seqs;
    double scale;
    const int32_t *key_lo, *key_hi; /* optional per-sequence key window */
    double *out, *lse;
    int64_t thread_index, num_threads;
    /* INT8 pages (NULL for bf16): codes [pages][P][Hkv][D], scales [pages][Hkv][P] */
    const int8_t *k_codes, *v_codes;
    const float *k_scales, *v_scales;
} kvo_attention_job;

/*
 * One (sequence, kv head): gather that head's keys and values through the block table
 * into contiguous fp64 rows (the oracle does on purpose the gather the GPU must avoid,
 * [PA] "Compute attention over scattered KV"), then, for every q head of the group and
 * every new token, the textbook softmax(q . K^T * scale) . V over the visible keys.
 */
static void attention_one_group(const kvo_attention_job *job, int64_t s, int64_t g,
                                double *k_rows, double *v_rows)
{
    const int64_t D = job->head_dim;
    const int64_t Hkv = job->kv_heads;
    const int64_t group = job->q_heads / job->kv_heads;
    const int64_t ctx = job->context_lens[s];
    const int64_t first = job->q_indptr[s];
    const int64_t q_len = job->q_indptr[s + 1] - first;

    /* Gather: key position p of this head -> k_rows[p*D .. p*D+D-1].  INT8 pages hold
     * x = scale * code ([TI] "INT8 cache"); the oracle forms that value exactly in fp64. */
    for (int64_t p = 0; p < ctx; ++p) {
        int64_t slot = kvo_slot_of_position(job->block_table, job->bt_stride, s, p,
                                            job->page_size);
        if (job->k_codes) {
            int64_t page = slot / job->page_size, off = slot % job->page_size;
            double ks = job->k_scales[(page * Hkv + g) * job->page_size + off];
            double vs = job->v_scales[(page * Hkv + g) * job->page_size + off];
            const int8_t *kc = job->k_codes + (slot * Hkv + g) * D;
            const int8_t *vc = job->v_codes + (slot * Hkv + g) * D;
            for (int64_t d = 0; d < D; ++d) {
                k_rows[p * D + d] = ks * (double)kc[d];
                v_rows[p * D + d] = vs * (double)vc[d];
            }
            continue;
        }
        const uint16_t *kv = job->k_pool + (slot * Hkv + g) * D;
        const uint16_t *vv = job->v_pool + (slot * Hkv + g) * D;
        for (int64_t d = 0; d < D; ++d) {
            k_rows[p * D + d] = bf16_bits_to_double(kv[d]);
            v_rows[p * D + d] = bf16_bits_to_double(vv[d]);
        }
    }

    double *scores = (double *)malloc((size_t)(ctx > 0 ? ctx : 1) * sizeof(double));
    for (int64_t i = 0; i < q_len; ++i) {
        int64_t t = first + i;
        int64_t query_position = ctx - q_len + i;
        /* Visible keys: 0 .. query_position, optionally narrowed to [key_lo, key_hi). */
        int64_t lo = 0, hi = query_position + 1;
        if (job->key_lo && job->key_lo[s] > lo)
            lo = job->key_lo[s];
        if (job->key_hi && job->key_hi[s] < hi)
            hi = job->key_hi[s];
        for (int64_t j = 0; j < group; ++j) {
            int64_t h = g * group + j;
            const uint16_t *qv = job->q + (t * job->q_heads + h) * D;
            double *o = job->out + (t * job->q_heads + h) * D;
            double *lse = job->lse ? job->lse + t * job->q_heads + h : NULL;
            if (hi <= lo) {
                for (int64_t d = 0; d < D; ++d)
                    o[d] = 0.0;
                if (lse)
                    *lse = -INFINITY;
                continue;
            }
            /* x_p = (q . k_p) * scale */
            double max_score = -INFINITY;
            for (int64_t p = lo; p < hi; ++p) {
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    dot += bf16_bits_to_double(qv[d]) * k_rows[p * D + d];
                scores[p] = dot * job->scale;
                if (scores[p] > max_score)
                    max_score = scores[p];
            }
            /* w_p = exp(x_p - max);  o = sum_p w_p v_p / sum_p w_p */
            double denom = 0.0;
            for (int64_t d = 0; d < D; ++d)
                o[d] = 0.0;
            for (int64_t p = lo; p < hi; ++p) {
                double w = exp(scores[p] - max_score);
                denom += w;
                for (int64_t d = 0; d < D; ++d)
                    o[d] += w * v_rows[p * D + d];
            }
            for (int64_t d = 0; d < D; ++d)
                o[d] /= denom;
            if (lse)
                *lse = max_score + log(denom);
        }
    }
    free(scores);
}

static void *attention_worker(void *arg)
{
    const kvo_attention_job *job = (const kvo_attention_job *)arg;
    int64_t max_ctx = 0;
    for (int64_t s = 0; s < job->num_seqs; ++s)
        if (job->context_lens[s] > max_ctx)
            max_ctx = job->context_lens[s];
    size_t rows = (size_t)(max_ctx > 0 ? max_ctx : 1) * (size_t)job->head_dim;
    double *k_rows = (double *)malloc(rows * sizeof(double));
    double *v_rows = (double *)malloc(rows * sizeof(double));
    /* Work item w = s * kv_heads + g; thread k takes w = k, k + n, k + 2n, ... */
    int64_t items = job->num_seqs * job->kv_heads;
    for (int64_t w = job->thread_index; w < items; w += job->num_threads)
        attention_one_group(job, w / job->kv_heads, w % job->kv_heads, k_rows, v_rows);
    free(k_rows);
    free(v_rows);
    return NULL;
}

/*
 * Paged attention for decode (q_len = 1 per sequence) and for appended chunks
 * (q_len >= 1, causal over the cached prefix plus the chunk).
 *
 *   q            [T][q_heads][head_dim] bf16 bits, T = q_indptr[num_seqs]
 *   k_pool/v_pool [num_pages][page_size][kv_heads][head_dim] bf16 bits
 *   block_table  [num_seqs][bt_stride] int32 page ids
 *   context_lens [num_seqs], q_indptr [num_seqs + 1]
 *   key_lo/key_hi optional [num_seqs]: restrict keys to [key_lo, key_hi) (used to check
 *                split-K partials); NULL for the whole visible range
 *   out          [T][q_heads][head_dim] fp64;  lse [T][q_heads] fp64 or NULL
 *   num_threads  >= 1; threads take disjoint (sequence, kv head) items, so the result does
 *                not depend on it
 */
static void run_attention(kvo_attention_job base, int64_t num_threads)
{
    if (num_threads < 1)
        num_threads = 1;
    kvo_attention_job *jobs =
        (kvo_attention_job *)calloc((size_t)num_threads, sizeof(kvo_attention_job));
    pthread_t *threads = (pthread_t *)calloc((size_t)num_threads, sizeof(pthread_t));
    for (int64_t k = 0; k < num_threads; ++k) {
        jobs[k] = base;
        jobs[k].thread_index = k;
        jobs[k].num_threads = num_threads;
    }
    if (num_threads == 1) {
        attention_worker(&jobs[0]);
    } else {
        for (int64_t k = 0; k < num_threads; ++k)
            pthread_create(&threads[k], NULL, attention_worker, &jobs[k]);
        for (int64_t k = 0; k < num_threads; ++k)
            pthread_join(threads[k], NULL);
    }
    free(threads);
    free(jobs);
}

void kvo_attention(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                   int64_t page_size, int64_t kv_heads, int64_t head_dim,
                   const int32_t *block_table, int64_t bt_stride,
                   const int32_t *context_lens, const int32_t *q_indptr, int64_t num_seqs,
                   int64_t q_heads, double scale, const int32_t *key_lo,
                   const int32_t *key_hi, double *out, double *lse, int64_t num_threads)
{
    kvo_attention_job j = {q,         k_pool,       v_pool,   page_size, kv_heads,
                           head_dim,  q_heads,      block_table, bt_stride,
                           context_lens, q_indptr,  num_seqs, scale,     key_lo,
                           key_hi,    out,          lse,      0,         1,
                           NULL,      NULL,         NULL,     NULL};
    run_attention(j, num_threads);
}

/*
 * The same attention over INT8 pages ([TI] "INT8 cache"): position p of kv head g holds
 * codes c (int8) and one scale s, and stands for the vector s * c.  Attention in the pages'
 * form (the key scale multiplying its score, the value scale its probability) equals the
 * plain attention over those vectors, which is what the oracle computes.
 *   k_codes/v_codes  [num_pages][page_size][kv_heads][head_dim] int8
 *   k_scales/v_scales [num_pages][kv_heads][page_size] fp32
 */
void kvo_attention_int8(const uint16_t *q, const int8_t *k_codes, const int8_t *v_codes,
                        const float *k_scales, const float *v_scales, int64_t page_size,
                        int64_t kv_heads, int64_t head_dim, const int32_t *block_table,
                        int64_t bt_stride, const int32_t *context_lens,
                        const int32_t *q_indptr, int64_t num_seqs, int64_t q_heads,
                        double scale, const int32_t *key_lo, const int32_t *key_hi,
                        double *out, double *lse, int64_t num_threads)
{
    kvo_attention_job j = {q,         NULL,         NULL,     page_size, kv_heads,
                           head_dim,  q_heads,      block_table, bt_stride,
                           context_lens, q_indptr,  num_seqs, scale,     key_lo,
                           key_hi,    out,          lse,      0,         1,
                           k_codes,   v_codes,      k_scales, v_scales};
    run_attention(j, num_threads);
}

/*
 * Merge of split partials by log-sum-exp, written out from its definition: partial j
 * holds o_j (normalised over its own keys) and lse_j; the union of the splits has
 * lse = log(sum_j exp(lse_j)) and o = sum_j exp(lse_j - lse) o_j.  Splits with
 * lse_j = -inf hold no key and add nothing; if every split is empty, o = 0.
 *   partial_o   [rows][num_splits][head_dim] fp64
 *   partial_lse [rows][num_splits] fp64
 */
void kvo_merge(const double *partial_o, const double *partial_lse, int64_t rows,
               int64_t num_splits, int64_t head_dim, double *out, double *lse_out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *l = partial_lse + r * num_splits;
        double m = -INFINITY;
        for (int64_t j = 0; j < num_splits; ++j)
            if (l[j] > m)
                m = l[j];
        double *o = out + r * head_dim;
        for (int64_t d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        if (m == -INFINITY) {
            if (lse_out)
                lse_out[r] = -INFINITY;
            continue;
        }
        double total = 0.0;
        for (int64_t j = 0; j < num_splits; ++j)
            total += exp(l[j] - m);
        double lse = m + log(total);
        for (int64_t j = 0; j < num_splits; ++j) {
            if (l[j] == -INFINITY)
                continue; /* an empty split holds no key: its o_j is not read at all */
            double w = exp(l[j] - lse);
            for (int64_t d = 0; d < head_dim; ++d)
                o[d] += w * partial_o[(r * num_splits + j) * head_dim + d];
        }
        if (lse_out)
            lse_out[r] = lse;
    }
}

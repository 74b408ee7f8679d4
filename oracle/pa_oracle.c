/*
 * pa_oracle.c -- CPU ORACLE for the paged-KV-cache decode path.
 *
 * THIS FILE IS TEST INFRASTRUCTURE.  Only the tests, the smoke check and the
 * bench's CPU-baseline leg may load it.  The product library never links,
 * loads or calls it, and it shares no code, header, table or helper with the
 * CUDA kernels.
 *
 * What it computes (plain definitions, written out with no blocking, fusion
 * or reordering beyond what the definitions state):
 *
 *   - half decode / encode: IEEE-754 binary16 and bfloat16, decoded from the
 *     bit layouts to double and encoded from double with round-to-nearest-even.
 *
 *   - cache write: for every new token t whose slot s = slot_mapping[t] is
 *     non-negative, the key row of every KV head is copied byte for byte to
 *     pool position (block s/B, head h, offset s%B) for block size B; same
 *     for the value.
 *     [Paged Attention: Managing the KV Cache Like Virtual Memory, "A paged KV
 *     cache, in code" (PagedLayer.update writes through blocks/offsets, and the
 *     closing note on the slot mapping that says where each token's keys and
 *     values go); Efficient Memory Management for LLM Serving with
 *     PagedAttention, "Kernel-Level Optimizations", 1. fused reshape and block
 *     write]
 *
 *   - block copy: for every layer and every (src, dst) pair, block dst of the
 *     K pool and of the V pool becomes a byte copy of block src.
 *
 *   - swap: the same byte copy between two pools (the GPU pool and the CPU
 *     swap space, in either direction): block dst of the destination pool
 *     becomes a copy of block src of the source pool.
 *     [Efficient Memory Management ..., "Kernel-Level Optimizations", 3. fused
 *     block copy; "Copy-on-write mechanism"]
 *
 *   - decode attention: for sequence s and query head h (KV head h / G with
 *     G = num_heads / num_kv_heads, consecutive grouping), token t of the
 *     context lives at block_tables[s][t/B], offset t%B.  With
 *     x_t = scale * sum_d q[d] k_t[d], the output is
 *        o = sum_t exp(x_t - m) v_t / sum_t exp(x_t - m),   m = max_t x_t,
 *     i.e. the standard attention equation (a_ij, o_i) with the caller's scale,
 *     evaluated in double, two passes (max, then sums).
 *     [Efficient Memory Management ..., "PagedAttention Algorithm": standard
 *     attention equation and its block-wise reformulation, which computes the
 *     same o_i; vLLM Internals, "PagedAttention: page tables, for KV"
 *     (resolve: divmod of the position by the block size, then a table
 *     lookup); Paged Attention: Managing the KV Cache ..., "Attention over
 *     scattered blocks" (row(): block, kv head, offset, dim addressing)]
 *
 *   - prefill (chunked prefill) attention: the i-th of a sequence's n new
 *     tokens, at position p = context_lens[s] - n + i, attends causally over
 *     positions 0 .. p: the decode attention of its query row over the first
 *     p + 1 tokens of the sequence.
 *
 *   - block-wise decode attention: the same output computed block by block
 *     with a per-block partial state (max, sum of exponentials, weighted sum of
 *     values) and a final merge, the block-wise form of the attention equation.
 *     It exists only so the tests can check that the block-wise form and the
 *     token-wise form agree.
 *
 * Layouts (all row-major, all caller-owned host memory):
 *   q           [num_seqs][num_heads][head_dim]                  16-bit codes
 *   k/v pools   [num_blocks][num_kv_heads][B][head_dim]           16-bit codes
 *
 * B (block_size) is the number of tokens per block, any positive value: the
 * method fixes it per cache, not per kernel [Efficient Memory Management ...,
 * "PagedAttention Algorithm": the KV cache is partitioned into blocks of B
 * tokens; Paged Attention: Managing the KV Cache ..., benchmark section: the
 * same attention swept over block sizes].
 *   block_tables[num_seqs][max_blocks_per_seq]                    int32
 *   context_lens[num_seqs]                                        int32
 *   out         [num_seqs][num_heads][head_dim]                   double
 *
 * Return codes: 0 = ok, 1 = invalid argument, 2 = block id out of range,
 * 3 = slot out of range, 4 = out of memory.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* ------------------------------------------------------------------------ */
/* 16-bit float codes <-> double, from the bit layouts.                       */
/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.                  */
/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.                  */
/* ------------------------------------------------------------------------ */

static void layout(int dtype, int *ebits, int *fbits, int *bias) {
    if (dtype == ORACLE_F16) { *ebits = 5; *fbits = 10; *bias = 15; }
    else                     { *ebits = 8; *fbits = 7;  *bias = 127; }
}

double pa_oracle_half_to_double(uint16_t code, int dtype) {
    int ebits, fbits, bias;
    layout(dtype, &ebits, &fbits, &bias);
    unsigned sign = (code >> 15) & 1u;
    unsigned e = (code >> fbits) & ((1u << ebits) - 1u);
    unsigned f = code & ((1u << fbits) - 1u);
    double mag;
    if (e == 0) {                                  /* zero or subnormal */
        mag = ldexp((double)f, 1 - bias - fbits);
    } else if (e == (1u << ebits) - 1u) {          /* inf or nan */
        mag = (f == 0) ? INFINITY : NAN;
    } else {                                       /* normal */
        mag = ldexp((double)((1u << fbits) | f), (int)e - bias - fbits);
    }
    return sign ? -mag : mag;
}

/* Round-to-nearest-even encode of a double into a 16-bit code. */
uint16_t pa_oracle_double_to_half(double x, int dtype) {
    int ebits, fbits, bias;
    layout(dtype, &ebits, &fbits, &bias);
    const unsigned emax_code = (1u << ebits) - 1u;
    uint16_t sign = (uint16_t)(signbit(x) ? 0x8000u : 0u);
    if (isnan(x)) {
        /* quiet nan: all-ones exponent, top fraction bit set */
        return (uint16_t)(sign | (emax_code << fbits) | (1u << (fbits - 1)));
    }
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | (emax_code << fbits));
    if (a == 0.0) return sign;

    /* quantum (spacing of representable values) at a's binade */
    const int emin = 1 - bias;                     /* smallest normal exponent */
    int e2;
    (void)frexp(a, &e2);                           /* a = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                                /* a in [2^e, 2^(e+1)) */
    if (e < emin) e = emin;                        /* subnormal range: fixed quantum */
    double q = ldexp(1.0, e - fbits);
    double n = a / q;                              /* exact: power-of-two scaling */
    double r = nearbyint(n);                       /* default mode: ties to even */
    double v = r * q;                              /* the rounded magnitude, exact */

    double maxfinite = ldexp((double)((2u << fbits) - 1u), (int)emax_code - 1 - bias - fbits);
    if (v > maxfinite) return (uint16_t)(sign | (emax_code << fbits));

    if (v < ldexp(1.0, emin)) {                    /* subnormal (or rounded to 0) */
        unsigned frac = (unsigned)(v / ldexp(1.0, emin - fbits));
        return (uint16_t)(sign | frac);
    }
    int ev2;
    double m = frexp(v, &ev2);                     /* v = m * 2^ev2 */
    int ev = ev2 - 1;                              /* v in [2^ev, 2^(ev+1)) */
    unsigned frac = (unsigned)((2.0 * m - 1.0) * (double)(1u << fbits));
    unsigned ecode = (unsigned)(ev + bias);
    return (uint16_t)(sign | (ecode << fbits) | frac);
}

void pa_oracle_decode_halves(const uint16_t *in, double *out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = pa_oracle_half_to_double(in[i], dtype);
}

void pa_oracle_encode_halves(const double *in, uint16_t *out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = pa_oracle_double_to_half(in[i], dtype);
}

/* ------------------------------------------------------------------------ */
/* Cache write: token t's K/V rows go to slot slot_mapping[t] of the pool.    */
/* ------------------------------------------------------------------------ */
int pa_oracle_cache_write(const uint16_t *key, const uint16_t *value,
                          uint16_t *k_cache, uint16_t *v_cache,
                          const int64_t *slot_mapping, int num_tokens,
                          int num_blocks, int num_kv_heads, int head_dim, int block_size) {
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0)
        return 1;
    int rc = 0;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;                              /* padding token: no slot */
        if (slot >= (int64_t)num_blocks * block_size) { rc = 3; continue; }
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim;
            memcpy(k_cache + dst, key + src, sizeof(uint16_t) * head_dim);
            memcpy(v_cache + dst, value + src, sizeof(uint16_t) * head_dim);
        }
    }
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Block copy: for each layer and pair, pool[dst] = pool[src] (K and V).      */
/* k_caches / v_caches are arrays of num_layers host pointers.               */
/* ------------------------------------------------------------------------ */
int pa_oracle_copy_blocks(uint16_t *const *k_caches, uint16_t *const *v_caches, int num_layers,
                          const int64_t *block_pairs, int num_pairs,
                          int num_blocks, int num_kv_heads, int head_dim, int block_size) {
    if (num_layers < 0 || num_pairs < 0 || num_blocks <= 0 || block_size <= 0) return 1;
    size_t block_elems = (size_t)num_kv_heads * block_size * head_dim;
    int rc = 0;
    for (int l = 0; l < num_layers; ++l) {
        for (int i = 0; i < num_pairs; ++i) {
            int64_t src = block_pairs[2 * i], dst = block_pairs[2 * i + 1];
            if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { rc = 2; continue; }
            memcpy(k_caches[l] + (size_t)dst * block_elems, k_caches[l] + (size_t)src * block_elems,
                   sizeof(uint16_t) * block_elems);
            memcpy(v_caches[l] + (size_t)dst * block_elems, v_caches[l] + (size_t)src * block_elems,
                   sizeof(uint16_t) * block_elems);
        }
    }
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Swap: for each layer and pair, dst_pool[dst] = src_pool[src] (K and V),    */
/* between two pools (GPU pool and CPU swap space, either way).               */
/* [Efficient Memory Management ..., "Scheduling and Preemption", swapping:   */
/* evicted blocks are copied to CPU RAM and copied back when the sequence     */
/* resumes, with a CPU block allocator mirroring the GPU one]                 */
/* ------------------------------------------------------------------------ */
int pa_oracle_swap_blocks(uint16_t *const *dst_k, uint16_t *const *dst_v,
                          const uint16_t *const *src_k, const uint16_t *const *src_v,
                          int num_layers, const int64_t *block_pairs, int num_pairs,
                          int num_dst_blocks, int num_src_blocks, int num_kv_heads, int head_dim,
                          int block_size) {
    if (num_layers < 0 || num_pairs < 0 || num_dst_blocks <= 0 || num_src_blocks <= 0 ||
        block_size <= 0)
        return 1;
    size_t block_elems = (size_t)num_kv_heads * block_size * head_dim;
    int rc = 0;
    for (int l = 0; l < num_layers; ++l) {
        for (int i = 0; i < num_pairs; ++i) {
            int64_t src = block_pairs[2 * i], dst = block_pairs[2 * i + 1];
            if (src < 0 || src >= num_src_blocks || dst < 0 || dst >= num_dst_blocks) { rc = 2; continue; }
            memcpy(dst_k[l] + (size_t)dst * block_elems, src_k[l] + (size_t)src * block_elems,
                   sizeof(uint16_t) * block_elems);
            memcpy(dst_v[l] + (size_t)dst * block_elems, src_v[l] + (size_t)src * block_elems,
                   sizeof(uint16_t) * block_elems);
        }
    }
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Decode attention.                                                          */
/* ------------------------------------------------------------------------ */
typedef struct {
    double *out;
    double *weights;                 /* optional [num_seqs][num_heads][max_ctx] */
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    int max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks, block_size;
    int max_ctx, dtype, blockwise;
    double scale;
    int nthreads, tid;
    int rc;
} attn_job;

/* Address of token t's row (K or V) of KV head hk in sequence s, or NULL if
 * the table entry is out of range. */
static const uint16_t *token_row(const attn_job *J, const uint16_t *pool, int s, int hk, int t) {
    const int B = J->block_size;
    int32_t blk = J->block_tables[(size_t)s * J->max_blocks_per_seq + t / B];
    if (blk < 0 || blk >= J->num_blocks) return NULL;
    int off = t % B;
    return pool + (((size_t)blk * J->num_kv_heads + hk) * B + off) * J->head_dim;
}

/* Token-wise form: two passes, scores first, then max, exp, sums, for the
 * query row qrow (query head h) of sequence s over its first L tokens. */
static int attend_rows(const attn_job *J, int s, int h, const uint16_t *qrow, int L, double *x,
                       double *qd, double *o, double *weights_row) {
    const int D = J->head_dim, G = J->num_heads / J->num_kv_heads, hk = h / G;
    for (int d = 0; d < D; ++d) qd[d] = pa_oracle_half_to_double(qrow[d], J->dtype);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (L <= 0) return 0;                                   /* empty context: zeros */

    for (int t = 0; t < L; ++t) {                           /* scores */
        const uint16_t *krow = token_row(J, J->k_cache, s, hk, t);
        if (!krow) return 2;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * pa_oracle_half_to_double(krow[d], J->dtype);
        x[t] = J->scale * dot;
    }
    double m = x[0];                                        /* pass 1: max */
    for (int t = 1; t < L; ++t) if (x[t] > m) m = x[t];
    double Z = 0.0;                                         /* pass 2: exp, sums */
    for (int t = 0; t < L; ++t) {
        double w = exp(x[t] - m);
        x[t] = w;
        Z += w;
    }
    for (int t = 0; t < L; ++t) {
        const uint16_t *vrow = token_row(J, J->v_cache, s, hk, t);
        if (!vrow) return 2;
        for (int d = 0; d < D; ++d) o[d] += x[t] * pa_oracle_half_to_double(vrow[d], J->dtype);
    }
    for (int d = 0; d < D; ++d) o[d] /= Z;
    if (weights_row)
        for (int t = 0; t < L; ++t) weights_row[t] = x[t] / Z;
    return 0;
}

/* Decode: sequence s's one query row per head over its context_lens[s] tokens. */
static int attend_tokenwise(const attn_job *J, int s, int h, double *x, double *qd, double *o) {
    const uint16_t *qrow = J->q + ((size_t)s * J->num_heads + h) * J->head_dim;
    double *w = J->weights ? J->weights + ((size_t)s * J->num_heads + h) * J->max_ctx : NULL;
    return attend_rows(J, s, h, qrow, J->context_lens[s], x, qd, o, w);
}

/* Block-wise form: each logical block j yields (m_j, l_j, acc_j) over its own
 * tokens; the merge rescales every partial to the global max. */
static int attend_blockwise(const attn_job *J, int s, int h, double *x, double *qd, double *o,
                            double *bm, double *bl, double *bacc) {
    const int D = J->head_dim, G = J->num_heads / J->num_kv_heads, hk = h / G;
    const int L = J->context_lens[s];
    const uint16_t *qrow = J->q + ((size_t)s * J->num_heads + h) * D;
    for (int d = 0; d < D; ++d) qd[d] = pa_oracle_half_to_double(qrow[d], J->dtype);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (L <= 0) return 0;
    const int B = J->block_size;
    const int nb = (L + B - 1) / B;
    for (int j = 0; j < nb; ++j) {
        int t0 = j * B, t1 = t0 + B < L ? t0 + B : L;
        double mj = -INFINITY;
        for (int t = t0; t < t1; ++t) {
            const uint16_t *krow = token_row(J, J->k_cache, s, hk, t);
            if (!krow) return 2;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qd[d] * pa_oracle_half_to_double(krow[d], J->dtype);
            x[t - t0] = J->scale * dot;
            if (x[t - t0] > mj) mj = x[t - t0];
        }
        double lj = 0.0;
        double *accj = bacc + (size_t)j * D;
        for (int d = 0; d < D; ++d) accj[d] = 0.0;
        for (int t = t0; t < t1; ++t) {
            double w = exp(x[t - t0] - mj);
            lj += w;
            const uint16_t *vrow = token_row(J, J->v_cache, s, hk, t);
            if (!vrow) return 2;
            for (int d = 0; d < D; ++d) accj[d] += w * pa_oracle_half_to_double(vrow[d], J->dtype);
        }
        bm[j] = mj;
        bl[j] = lj;
    }
    double M = bm[0];
    for (int j = 1; j < nb; ++j) if (bm[j] > M) M = bm[j];
    double Lsum = 0.0;
    for (int j = 0; j < nb; ++j) {
        double c = exp(bm[j] - M);
        Lsum += bl[j] * c;
        for (int d = 0; d < D; ++d) o[d] += bacc[(size_t)j * D + d] * c;
    }
    for (int d = 0; d < D; ++d) o[d] /= Lsum;
    return 0;
}

static void *attn_worker(void *arg) {
    attn_job *J = (attn_job *)arg;
    const int D = J->head_dim;
    const int B = J->block_size;
    const int maxnb = (J->max_ctx + B - 1) / B + 1;
    double *x = (double *)malloc(sizeof(double) * (size_t)(J->max_ctx > B ? J->max_ctx : B));
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *bm = (double *)malloc(sizeof(double) * (size_t)maxnb);
    double *bl = (double *)malloc(sizeof(double) * (size_t)maxnb);
    double *bacc = J->blockwise ? (double *)malloc(sizeof(double) * (size_t)maxnb * D) : NULL;
    if (!x || !qd || !bm || !bl || (J->blockwise && !bacc)) {
        J->rc = 4;
    } else {
        const long total = (long)J->num_seqs * J->num_heads;
        for (long i = J->tid; i < total; i += J->nthreads) {   /* static striding over (s, h) */
            int s = (int)(i / J->num_heads), h = (int)(i % J->num_heads);
            double *o = J->out + (size_t)i * D;
            int rc = J->blockwise ? attend_blockwise(J, s, h, x, qd, o, bm, bl, bacc)
                                  : attend_tokenwise(J, s, h, x, qd, o);
            if (rc && !J->rc) J->rc = rc;
        }
    }
    free(x); free(qd); free(bm); free(bl); free(bacc);
    return NULL;
}

static int run_attention(double *out, double *weights, const uint16_t *q,
                         const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, int num_seqs, int num_heads,
                         int num_kv_heads, int head_dim, int num_blocks, int block_size,
                         double scale, int dtype, int nthreads, int blockwise) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_heads % num_kv_heads != 0 || num_blocks <= 0 || block_size <= 0 ||
        max_blocks_per_seq < 0 ||
        (dtype != ORACLE_F16 && dtype != ORACLE_BF16))
        return 1;
    int max_ctx = 0;
    for (int s = 0; s < num_seqs; ++s) {
        if (context_lens[s] < 0 || (int64_t)context_lens[s] > (int64_t)max_blocks_per_seq * block_size)
            return 1;
        if (context_lens[s] > max_ctx) max_ctx = context_lens[s];
    }
    if (nthreads < 1) nthreads = 1;
    attn_job *jobs = (attn_job *)calloc((size_t)nthreads, sizeof(attn_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 4; }
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        attn_job J = {out, weights, q, k_cache, v_cache, block_tables, context_lens,
                      max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks,
                      block_size, max_ctx, dtype, blockwise, scale, nthreads, i, 0};
        jobs[i] = J;
    }
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, attn_worker, &jobs[i]) != 0) break;
        started = i;
    }
    /* threads that could not be started: run their share here */
    for (int i = started + 1; i < nthreads; ++i) attn_worker(&jobs[i]);
    attn_worker(&jobs[0]);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) if (jobs[i].rc && !rc) rc = jobs[i].rc;
    free(jobs); free(th);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Prefill (chunked prefill) attention.                                       */
/* Sequence s has n_s = query_start_loc[s+1] - query_start_loc[s] new tokens, */
/* already written to the cache as its last n_s positions, so its i-th new    */
/* token sits at position p = context_lens[s] - n_s + i and attends causally  */
/* over positions 0 .. p: the decode attention of that row over the first     */
/* p + 1 tokens.  [Efficient Memory Management ..., "End-to-End Decoding":    */
/* the prompt phase computes the KV cache of all prompt tokens and attends    */
/* over them in one pass; vLLM Internals ..., the scheduler's chunked prefill  */
/* (a prompt processed a token budget at a time)]                              */
/* ------------------------------------------------------------------------ */
typedef struct {
    attn_job base;
    const int32_t *qsl;          /* [num_seqs + 1] */
    int num_tokens;
} prefill_job;

static void *prefill_worker(void *arg) {
    prefill_job *P = (prefill_job *)arg;
    attn_job *J = &P->base;
    const int D = J->head_dim;
    double *x = (double *)malloc(sizeof(double) * (size_t)(J->max_ctx > 1 ? J->max_ctx : 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    if (!x || !qd) {
        J->rc = 4;
    } else {
        const long total = (long)P->num_tokens * J->num_heads;
        for (long i = J->tid; i < total; i += J->nthreads) {
            const int t = (int)(i / J->num_heads), h = (int)(i % J->num_heads);
            int s = 0;
            while (s + 1 < J->num_seqs && P->qsl[s + 1] <= t) ++s;     /* t's sequence */
            const int n = P->qsl[s + 1] - P->qsl[s];
            const int L = J->context_lens[s] - n + (t - P->qsl[s]) + 1;
            const uint16_t *qrow = J->q + ((size_t)t * J->num_heads + h) * D;
            int rc = attend_rows(J, s, h, qrow, L, x, qd, J->out + (size_t)i * D, NULL);
            if (rc && !J->rc) J->rc = rc;
        }
    }
    free(x);
    free(qd);
    return NULL;
}

int pa_oracle_prefill_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                                const uint16_t *v_cache, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *query_start_loc,
                                const int32_t *context_lens, int num_seqs, int num_tokens,
                                int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                                int block_size, double scale, int dtype, int nthreads) {
    if (num_seqs < 0 || num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || num_heads % num_kv_heads != 0 || num_blocks <= 0 || block_size <= 0 ||
        max_blocks_per_seq < 0 || (dtype != ORACLE_F16 && dtype != ORACLE_BF16))
        return 1;
    if (query_start_loc[0] != 0 || query_start_loc[num_seqs] != num_tokens) return 1;
    int max_ctx = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int n = query_start_loc[s + 1] - query_start_loc[s];
        if (n < 0 || context_lens[s] < n ||
            (int64_t)context_lens[s] > (int64_t)max_blocks_per_seq * block_size)
            return 1;
        if (context_lens[s] > max_ctx) max_ctx = context_lens[s];
    }
    if (nthreads < 1) nthreads = 1;
    prefill_job *jobs = (prefill_job *)calloc((size_t)nthreads, sizeof(prefill_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 4; }
    for (int i = 0; i < nthreads; ++i) {
        attn_job J = {out, NULL, q, k_cache, v_cache, block_tables, context_lens,
                      max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks,
                      block_size, max_ctx, dtype, 0, scale, nthreads, i, 0};
        jobs[i].base = J;
        jobs[i].qsl = query_start_loc;
        jobs[i].num_tokens = num_tokens;
    }
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, prefill_worker, &jobs[i]) != 0) break;
        started = i;
    }
    for (int i = started + 1; i < nthreads; ++i) prefill_worker(&jobs[i]);
    prefill_worker(&jobs[0]);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) if (jobs[i].base.rc && !rc) rc = jobs[i].base.rc;
    free(jobs);
    free(th);
    return rc;
}

int pa_oracle_decode_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                               const uint16_t *v_cache, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                               int block_size, double scale, int dtype, int nthreads) {
    return run_attention(out, NULL, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                         context_lens, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks,
                         block_size, scale, dtype, nthreads, 0);
}

/* Same as above, also returning the normalised weights a_t = w_t / Z in
 * weights[s][h][t] (row length max_ctx = max over s of context_lens[s]). */
int pa_oracle_attention_weights(double *out, double *weights, const uint16_t *q,
                                const uint16_t *k_cache, const uint16_t *v_cache,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, int num_seqs, int num_heads,
                                int num_kv_heads, int head_dim, int num_blocks, int block_size,
                                double scale, int dtype) {
    return run_attention(out, weights, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                         context_lens, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks,
                         block_size, scale, dtype, 1, 0);
}

int pa_oracle_decode_attention_blockwise(double *out, const uint16_t *q, const uint16_t *k_cache,
                                         const uint16_t *v_cache, const int32_t *block_tables,
                                         int max_blocks_per_seq, const int32_t *context_lens,
                                         int num_seqs, int num_heads, int num_kv_heads,
                                         int head_dim, int num_blocks, int block_size,
                                         double scale, int dtype, int nthreads) {
    return run_attention(out, NULL, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                         context_lens, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks,
                         block_size, scale, dtype, nthreads, 1);
}

/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for split-KV paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load, link or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline /
 * reference leg do.  It shares no code, header, table or constant with the CUDA
 * library; the two meet only through the seeded input generators.
 *
 * What it computes is the plain definition of attention over keys gathered
 * through a per-request block table, with no splitting, blocking or fusion:
 * flash-decoding's split-KV decomposition reaches this same result up to the
 * rounding order, so the definition itself is the oracle.  Every value is
 * decoded exactly to double and all arithmetic is done in double.
 *
 * Sources (page title, then the section the step follows):
 *  - "vllm.models.flint.ops.decode_attention", flint_decode_attention
 *    parameters: q [B, num_heads, 128]; kv_cache [num_blocks, num_kv_heads,
 *    page, 256] with K in [..., :128] and V in [..., 128:]; seq_lens counts the
 *    KV positions including the current token and 0 writes zeros; window
 *    attends to the last `window` positions; sinks are per-head fp32 logits.
 *  - same page, module description ("Numerics ..."): the sink adds
 *    exp2(sink*log2(e) - m*c) to the final denominator with c = scale*log2(e),
 *    i.e. exp(sink - scale*m): the sink is a natural-log logit that is NOT
 *    multiplied by the softmax scale.
 *  - "vllm.v1.attention.ops.triton_decode_attention", decode_attention_fwd_verify
 *    parameters: q [B*qlen, H, Lk] with a request's verify tokens contiguous;
 *    paged latent cache [num_pages, page, 1, Lk]; V is k_buffer[..., :Lv];
 *    lse is the natural-log LSE, -inf for rows with no key; row limit
 *    max(min(L - qlen + 1 + t, L_real), 0); k_scale dequantises an FP8 cache.
 *  - "Atencion paginada" (transformers), decode path: block_table row b holds
 *    the physical page of each logical page of request b; -1 marks unassigned
 *    entries; key j of request b lives at page block_table[b][j / page],
 *    slot j % page.
 *
 * Readings taken where the pages are silent:
 *  - lse excludes the sink (key-only log-sum-exp).  A sink-inclusive value would
 *    be finite for a row with no key, which the verify page rules out.
 *  - an MLA row with no key writes zeros, as the GQA path does.
 *  - window <= 0 means "no window"; otherwise keys [max(L - window, 0), L).
 *  - FP8 is OCP float8 e4m3 "fn": bias 7, 3 mantissa bits, subnormals,
 *    no infinities, S.1111.111 is NaN.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_PAGE -2
#define ORACLE_ERR_NOMEM -3

/* bfloat16: the upper half of an IEEE-754 binary32 (1 sign, 8 exponent,
 * 7 stored mantissa bits).  Decoding is exact: place the 16 bits in the high
 * half of a binary32 and widen. */
double pkv_oracle_bf16_to_f64(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* float8 e4m3 (OCP "fn" variant), decoded from the bit fields:
 *   s eeee mmm, bias 7.  e == 0: subnormal m/8 * 2^-6.  e == 15 and m == 7: NaN.
 *   otherwise (1 + m/8) * 2^(e - 7).  There is no infinity; max is 448. */
double pkv_oracle_e4m3_to_f64(uint8_t bits) {
    int s = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xF;
    int m = bits & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* ------------------------------------------------------------------------- */
/* GQA paged decode                                                           */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *q;
    int64_t q_sb, q_sh; /* element strides of q [B, Hq, D], last dim contiguous */
    const uint16_t *kv;
    int64_t kv_sblk, kv_sh, kv_stok; /* strides of kv [num_blocks, Hkv, P, 2D] */
    int64_t num_blocks;
    const int32_t *bt;
    int64_t bt_sb, max_blocks;
    const int32_t *seq_lens;
    const float *sinks; /* [Hq] or NULL */
    int window;
    double scale;
    int page_size, B, Hq, Hkv, D;
    const int64_t *rows; /* row = b * Hq + h; NULL means all B*Hq rows */
    int64_t nrows;
    double *out; /* [nrows, D] */
    double *lse; /* [nrows] */
    int status;
} gqa_job;

/* One output row of GQA decode: query head h of request b against kv head
 * h / (Hq / Hkv), over keys [s, L) gathered through the block table. */
static int gqa_row(const gqa_job *a, int64_t row, double *out, double *lse) {
    const int D = a->D, P = a->page_size;
    const int b = (int)(row / a->Hq), h = (int)(row % a->Hq);
    const int g = h / (a->Hq / a->Hkv);
    const int L = a->seq_lens[b];
    int s = 0;
    if (a->window > 0 && L > a->window) s = L - a->window;
    const int n = L > s ? L - s : 0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    if ((int64_t)((L + P - 1) / P) > a->max_blocks) return ORACLE_ERR_PAGE;

    double *x = (double *)malloc(sizeof(double) * (size_t)n);
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    const uint16_t **vrow = (const uint16_t **)malloc(sizeof(uint16_t *) * (size_t)n);
    if (!x || !qd || !vrow) {
        free(x); free(qd); free(vrow);
        return ORACLE_ERR_NOMEM;
    }
    const uint16_t *qrow = a->q + (int64_t)b * a->q_sb + (int64_t)h * a->q_sh;
    for (int d = 0; d < D; ++d) qd[d] = pkv_oracle_bf16_to_f64(qrow[d]);

    /* gather + scores */
    for (int j = s; j < L; ++j) {
        const int32_t page = a->bt[(int64_t)b * a->bt_sb + j / P];
        const int slot = j % P;
        if (page < 0 || (int64_t)page >= a->num_blocks) {
            free(x); free(qd); free(vrow);
            return ORACLE_ERR_PAGE;
        }
        const uint16_t *krow = a->kv + (int64_t)page * a->kv_sblk +
                               (int64_t)g * a->kv_sh + (int64_t)slot * a->kv_stok;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * pkv_oracle_bf16_to_f64(krow[d]);
        x[j - s] = a->scale * dot;
        vrow[j - s] = krow + D; /* V occupies [..., D:2D] of the same token row */
    }
    /* dense softmax */
    double M = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (x[i] > M) M = x[i];
    double Z = 0.0;
    for (int i = 0; i < n; ++i) Z += exp(x[i] - M);
    double den = Z;
    if (a->sinks) den += exp((double)a->sinks[h] - M);
    for (int i = 0; i < n; ++i) {
        const double w = exp(x[i] - M) / den;
        for (int d = 0; d < D; ++d) out[d] += w * pkv_oracle_bf16_to_f64(vrow[i][d]);
    }
    *lse = M + log(Z);
    free(x); free(qd); free(vrow);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* MLA causal verify                                                          */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *q;
    int64_t q_sr, q_sh; /* strides of q [B*qlen, H, Lk] */
    const uint8_t *cache; /* bf16 (2 bytes) or e4m3 (1 byte) elements */
    int fp8;
    const uint8_t *q8;       /* or: e4m3 query codes [r, h, Lk] (q ignored) */
    const float *q8_scale;   /* [r, h]: the query is code value * scale */
    int64_t q8_sr, q8_sh, qs_sr;
    int64_t c_spage, c_stok; /* element strides of the cache [num_pages, P, 1, Lk] */
    int64_t num_pages;
    const int32_t *bt;
    int64_t bt_sb, max_blocks;
    const int32_t *seq_lens, *real_seq_lens; /* real may be NULL */
    int qlen;
    double scale, k_scale;
    int page_size, B, H, Lk, Lv;
    const int64_t *rows; /* row = r * H + h, r = b * qlen + t */
    int64_t nrows;
    double *out; /* [nrows, Lv] */
    double *lse;
    int status;
} mla_job;

static double cache_elem(const mla_job *a, int64_t idx) {
    if (a->fp8) return pkv_oracle_e4m3_to_f64(a->cache[idx]) * a->k_scale;
    uint16_t bits;
    memcpy(&bits, a->cache + 2 * idx, 2);
    return pkv_oracle_bf16_to_f64(bits);
}

/* One output row of MLA verify: head h of verify token t of request b, over
 * keys [0, lim) with lim = max(min(L - qlen + 1 + t, L_real), 0).  The single
 * latent head serves every query head; V is the first Lv dims of K. */
static int mla_row(const mla_job *a, int64_t row, double *out, double *lse) {
    const int Lk = a->Lk, Lv = a->Lv, P = a->page_size;
    const int64_t r = row / a->H;
    const int h = (int)(row % a->H);
    const int b = (int)(r / a->qlen), t = (int)(r % a->qlen);
    const int L = a->seq_lens[b];
    const int Lr = a->real_seq_lens ? a->real_seq_lens[b] : L;
    int lim = L - a->qlen + 1 + t;
    if (Lr < lim) lim = Lr;
    if (lim < 0) lim = 0;
    for (int d = 0; d < Lv; ++d) out[d] = 0.0;
    if (lim == 0) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    if ((int64_t)((lim + P - 1) / P) > a->max_blocks) return ORACLE_ERR_PAGE;

    double *x = (double *)malloc(sizeof(double) * (size_t)lim);
    double *qd = (double *)malloc(sizeof(double) * (size_t)Lk);
    int64_t *kbase = (int64_t *)malloc(sizeof(int64_t) * (size_t)lim);
    if (!x || !qd || !kbase) {
        free(x); free(qd); free(kbase);
        return ORACLE_ERR_NOMEM;
    }
    if (a->q8) {
        const uint8_t *c8 = a->q8 + r * a->q8_sr + (int64_t)h * a->q8_sh;
        const double sq = (double)a->q8_scale[r * a->qs_sr + h];
        for (int d = 0; d < Lk; ++d) qd[d] = pkv_oracle_e4m3_to_f64(c8[d]) * sq;
    } else {
        const uint16_t *qrow = a->q + r * a->q_sr + (int64_t)h * a->q_sh;
        for (int d = 0; d < Lk; ++d) qd[d] = pkv_oracle_bf16_to_f64(qrow[d]);
    }
    for (int j = 0; j < lim; ++j) {
        const int32_t page = a->bt[(int64_t)b * a->bt_sb + j / P];
        if (page < 0 || (int64_t)page >= a->num_pages) {
            free(x); free(qd); free(kbase);
            return ORACLE_ERR_PAGE;
        }
        kbase[j] = (int64_t)page * a->c_spage + (int64_t)(j % P) * a->c_stok;
        double dot = 0.0;
        for (int d = 0; d < Lk; ++d) dot += qd[d] * cache_elem(a, kbase[j] + d);
        x[j] = a->scale * dot;
    }
    double M = -INFINITY;
    for (int j = 0; j < lim; ++j)
        if (x[j] > M) M = x[j];
    double Z = 0.0;
    for (int j = 0; j < lim; ++j) Z += exp(x[j] - M);
    for (int j = 0; j < lim; ++j) {
        const double w = exp(x[j] - M) / Z;
        for (int d = 0; d < Lv; ++d) out[d] += w * cache_elem(a, kbase[j] + d);
    }
    *lse = M + log(Z);
    free(x); free(qd); free(kbase);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Row-parallel driver: threads only split the independent output rows.       */
/* ------------------------------------------------------------------------- */

typedef struct {
    void *job;
    int kind; /* 0 = gqa, 1 = mla */
    int64_t next;
    pthread_mutex_t mu;
    int status;
} pool_t;

static void *worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        const int64_t i = p->next++;
        pthread_mutex_unlock(&p->mu);
        int rc;
        if (p->kind == 0) {
            gqa_job *a = (gqa_job *)p->job;
            if (i >= a->nrows) break;
            const int64_t row = a->rows ? a->rows[i] : i;
            rc = gqa_row(a, row, a->out + i * a->D, a->lse + i);
        } else {
            mla_job *a = (mla_job *)p->job;
            if (i >= a->nrows) break;
            const int64_t row = a->rows ? a->rows[i] : i;
            rc = mla_row(a, row, a->out + i * a->Lv, a->lse + i);
        }
        if (rc != ORACLE_OK) {
            pthread_mutex_lock(&p->mu);
            if (p->status == ORACLE_OK) p->status = rc;
            pthread_mutex_unlock(&p->mu);
        }
    }
    return NULL;
}

static int run_pool(void *job, int kind, int nthreads) {
    pool_t p;
    p.job = job;
    p.kind = kind;
    p.next = 0;
    p.status = ORACLE_OK;
    pthread_mutex_init(&p.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    pthread_t th[512];
    int started = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&th[started], NULL, worker, &p) == 0) ++started;
    worker(&p);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&p.mu);
    return p.status;
}

int pkv_oracle_gqa_decode(const uint16_t *q, int64_t q_sb, int64_t q_sh,
                          const uint16_t *kv, int64_t kv_sblk, int64_t kv_sh,
                          int64_t kv_stok, int64_t num_blocks, const int32_t *bt,
                          int64_t bt_sb, int64_t max_blocks, const int32_t *seq_lens,
                          const float *sinks, int window, double scale, int page_size,
                          int B, int Hq, int Hkv, int D, const int64_t *rows,
                          int64_t nrows, double *out, double *lse, int nthreads) {
    if (!q || !kv || !bt || !seq_lens || !out || !lse) return ORACLE_ERR_ARG;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || page_size <= 0)
        return ORACLE_ERR_ARG;
    if (!rows) nrows = (int64_t)B * Hq;
    for (int64_t i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= (int64_t)B * Hq) return ORACLE_ERR_ARG;
    gqa_job a = {q, q_sb, q_sh, kv, kv_sblk, kv_sh, kv_stok, num_blocks, bt, bt_sb,
                 max_blocks, seq_lens, sinks, window, scale, page_size, B, Hq, Hkv, D,
                 rows, nrows, out, lse, ORACLE_OK};
    return run_pool(&a, 0, nthreads);
}

int pkv_oracle_mla_verify(const uint16_t *q, int64_t q_sr, int64_t q_sh,
                          const void *cache, int fp8, int64_t c_spage, int64_t c_stok,
                          int64_t num_pages, const int32_t *bt, int64_t bt_sb,
                          int64_t max_blocks, const int32_t *seq_lens,
                          const int32_t *real_seq_lens, int qlen, double scale,
                          int page_size, double k_scale, int B, int H, int Lk, int Lv,
                          const int64_t *rows, int64_t nrows, double *out, double *lse,
                          int nthreads) {
    if (!q || !cache || !bt || !seq_lens || !out || !lse) return ORACLE_ERR_ARG;
    if (B < 0 || H <= 0 || qlen <= 0 || Lk <= 0 || Lv <= 0 || Lv > Lk || page_size <= 0)
        return ORACLE_ERR_ARG;
    if (!rows) nrows = (int64_t)B * qlen * H;
    for (int64_t i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= (int64_t)B * qlen * H) return ORACLE_ERR_ARG;
    mla_job a = {q, q_sr, q_sh, (const uint8_t *)cache, fp8, NULL, NULL, 0, 0, 0, c_spage,
                 c_stok, num_pages, bt, bt_sb, max_blocks, seq_lens, real_seq_lens, qlen, scale,
                 k_scale, page_size, B, H, Lk, Lv, rows, nrows, out, lse, ORACLE_OK};
    return run_pool(&a, 1, nthreads);
}

/* MLA verify with an e4m3-quantised query (see pkv_oracle_mla_quantize_q):
 * the query of (row r, head h) is code value x q_scale[r, h], exactly, and
 * everything else is pkv_oracle_mla_verify. */
int pkv_oracle_mla_verify_q8(const uint8_t *q8, int64_t q8_sr, int64_t q8_sh,
                             const float *q_scale, int64_t qs_sr, const void *cache, int fp8,
                             int64_t c_spage, int64_t c_stok, int64_t num_pages,
                             const int32_t *bt, int64_t bt_sb, int64_t max_blocks,
                             const int32_t *seq_lens, const int32_t *real_seq_lens, int qlen,
                             double scale, int page_size, double k_scale, int B, int H, int Lk,
                             int Lv, const int64_t *rows, int64_t nrows, double *out,
                             double *lse, int nthreads) {
    if (!q8 || !q_scale || !cache || !bt || !seq_lens || !out || !lse) return ORACLE_ERR_ARG;
    if (B < 0 || H <= 0 || qlen <= 0 || Lk <= 0 || Lv <= 0 || Lv > Lk || page_size <= 0)
        return ORACLE_ERR_ARG;
    if (!rows) nrows = (int64_t)B * qlen * H;
    for (int64_t i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= (int64_t)B * qlen * H) return ORACLE_ERR_ARG;
    mla_job a = {NULL, 0, 0, (const uint8_t *)cache, fp8, q8, q_scale, q8_sr, q8_sh, qs_sr,
                 c_spage, c_stok, num_pages, bt, bt_sb, max_blocks, seq_lens, real_seq_lens,
                 qlen, scale, k_scale, page_size, B, H, Lk, Lv, rows, nrows, out, lse,
                 ORACLE_OK};
    return run_pool(&a, 1, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Paged KV append.
 *
 * "Atencion paginada" (transformers), decode path, "Comportamiento de la
 * cache" and "Ejemplo": the decode kernel updates the paged cache in place;
 * the new token of a request with cache_seqlens[b] cached tokens goes to
 * logical position cache_seqlens[b], i.e. page block_table[b][pos / page],
 * slot pos % page (the example: 30 cached tokens -> block 2 slot 30; 32 ->
 * the second block, slot 0; 70 -> the third block, slot 6).
 * "vllm.models.flint.ops.decode_attention", flint_decode_attention
 * parameters: seq_lens counts the KV positions including the current token, so
 * with that convention the current token sits at seq_lens[b] - 1; for the MLA
 * verify rows (decode_attention_fwd_verify parameters: a request's qlen verify
 * tokens are its last qlen positions) row t of request b sits at
 * seq_lens[b] - qlen + t.
 *
 * Readings: a request with no position to write (seq_lens <= 0, or a verify row
 * before position 0) writes nothing; a position whose page entry is beyond the
 * table or outside the cache writes nothing and is counted in *skipped.  An FP8
 * cache stores e4m3(x / k_scale) with x / k_scale computed in fp32 (the
 * precision the library computes it in) and rounded to the nearest e4m3 value,
 * ties to even, saturating at +-448; -0 keeps its sign; NaN becomes 0x7F.
 */

/* float8 e4m3 "fn" encoding from the format's definition: normal values
 * (1 + m/8) 2^(e-7) for e = 1..15 (e = 15, m = 7 is NaN, so the largest is
 * 1.75 * 2^8 = 448), subnormals (m/8) 2^-6.  rint() rounds half to even in the
 * default rounding mode; every product below is exact in double. */
uint8_t pkv_oracle_f32_to_e4m3(float x) {
    const double v = (double)x;
    if (isnan(v)) return 0x7F;
    const int s = signbit(v) ? 1 : 0;
    const double a = fabs(v);
    int code;
    if (isinf(a)) {
        code = 0x7E; /* saturates like any value beyond 448 */
    } else if (a < ldexp(1.0, -6)) {
        const double q = rint(a * 512.0); /* multiples of 2^-9: 0 .. 8 */
        code = (q >= 8.0) ? (1 << 3) : (int)q;
    } else {
        int e;
        const double f = frexp(a, &e); /* a = f 2^e, f in [0.5, 1) */
        int E = e - 1;                 /* a = (2f) 2^E, 2f in [1, 2) */
        double q = rint(16.0 * f);     /* 8 * (2f): 8 .. 16 */
        if (q >= 16.0) {
            q = 8.0;
            E += 1;
        }
        if (E > 8 || (E == 8 && q > 14.0)) { /* beyond 448: saturate */
            E = 8;
            q = 14.0;
        }
        code = ((E + 7) << 3) | ((int)q - 8);
    }
    return (uint8_t)(code | (s << 7));
}

/* Query quantisation for the native-FP8 MLA path (a reading of the "Native-FP8
 * MLA MMA" step: the pages give no recipe): per (row, head), with the absolute
 * maximum a of the Lk bf16 elements, the scale is s = a / 448 computed in fp32
 * (round to nearest even; s = 1 when a = 0) and element d is stored as the
 * e4m3 code of q_d / s, the quotient computed in fp32 (the precision the
 * library computes it in), rounded as pkv_oracle_f32_to_e4m3 does.  The
 * dequantised query is code value x s. */
int pkv_oracle_mla_quantize_q(const uint16_t *q, int64_t q_sr, int64_t q_sh, int R, int H,
                              int Lk, uint8_t *codes, float *scales) {
    if (!q || !codes || !scales || R < 0 || H <= 0 || Lk <= 0) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < R; ++r)
        for (int h = 0; h < H; ++h) {
            const uint16_t *row = q + r * q_sr + (int64_t)h * q_sh;
            float amax = 0.0f;
            for (int d = 0; d < Lk; ++d) {
                const float v = (float)fabs(pkv_oracle_bf16_to_f64(row[d]));
                if (v > amax) amax = v;
            }
            const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[r * H + h] = sc;
            for (int d = 0; d < Lk; ++d) {
                const float x = (float)pkv_oracle_bf16_to_f64(row[d]) / sc;
                codes[(r * H + h) * (int64_t)Lk + d] = pkv_oracle_f32_to_e4m3(x);
            }
        }
    return ORACLE_OK;
}

static int append_slot(const int32_t *bt, int64_t bt_sb, int64_t max_blocks, int64_t num_blocks,
                       int64_t b, int64_t pos, int page_size, int64_t *blk, int64_t *slot) {
    const int64_t pg = pos / page_size;
    if (pg >= max_blocks) return 0;
    const int64_t id = bt[b * bt_sb + pg];
    if (id < 0 || id >= num_blocks) return 0;
    *blk = id;
    *slot = pos % page_size;
    return 1;
}

/* k, v: [B, Hkv, D] bf16 (row strides src_sb, src_sh); kv: [num_blocks, Hkv,
 * page, 2D] bf16 with K in [..., :D] and V in [..., D:]. */
int pkv_oracle_gqa_kv_append(const uint16_t *k, const uint16_t *v, int64_t src_sb, int64_t src_sh,
                             uint16_t *kv, int64_t kv_sblk, int64_t kv_sh, int64_t kv_stok,
                             int64_t num_blocks, const int32_t *bt, int64_t bt_sb,
                             int64_t max_blocks, const int32_t *seq_lens, int page_size,
                             int64_t B, int64_t Hkv, int64_t D, int64_t *skipped) {
    if (!k || !v || !kv || !bt || !seq_lens || page_size <= 0 || !skipped) return ORACLE_ERR_ARG;
    *skipped = 0;
    for (int64_t b = 0; b < B; ++b) {
        const int64_t L = seq_lens[b];
        if (L <= 0) continue;
        int64_t blk, slot;
        if (!append_slot(bt, bt_sb, max_blocks, num_blocks, b, L - 1, page_size, &blk, &slot)) {
            ++*skipped;
            continue;
        }
        for (int64_t h = 0; h < Hkv; ++h) {
            uint16_t *dst = kv + blk * kv_sblk + h * kv_sh + slot * kv_stok;
            const uint16_t *ks = k + b * src_sb + h * src_sh;
            const uint16_t *vs = v + b * src_sb + h * src_sh;
            for (int64_t d = 0; d < D; ++d) {
                dst[d] = ks[d];
                dst[D + d] = vs[d];
            }
        }
    }
    return ORACLE_OK;
}

/* latent: [B*qlen, Lk] bf16 (row stride lat_sr); cache: [num_pages, page, 1,
 * Lk] bf16 (fp8 = 0) or e4m3 bytes (fp8 = 1); k_scale: the fp32 scale (FP8). */
int pkv_oracle_mla_kv_append(const uint16_t *lat, int64_t lat_sr, void *cache, int fp8,
                             int64_t c_spage, int64_t c_stok, int64_t num_pages, const int32_t *bt,
                             int64_t bt_sb, int64_t max_blocks, const int32_t *seq_lens, int qlen,
                             int page_size, float k_scale, int64_t B, int64_t Lk,
                             int64_t *skipped) {
    if (!lat || !cache || !bt || !seq_lens || page_size <= 0 || qlen < 1 || !skipped)
        return ORACLE_ERR_ARG;
    *skipped = 0;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t t = 0; t < qlen; ++t) {
            const int64_t pos = (int64_t)seq_lens[b] - qlen + t;
            if (pos < 0) continue;
            int64_t pg, slot;
            if (!append_slot(bt, bt_sb, max_blocks, num_pages, b, pos, page_size, &pg, &slot)) {
                ++*skipped;
                continue;
            }
            const uint16_t *src = lat + (b * qlen + t) * lat_sr;
            const int64_t at = pg * c_spage + slot * c_stok;
            for (int64_t d = 0; d < Lk; ++d) {
                if (fp8) {
                    const float x = (float)pkv_oracle_bf16_to_f64(src[d]);
                    ((uint8_t *)cache)[at + d] = pkv_oracle_f32_to_e4m3(x / k_scale);
                } else {
                    ((uint16_t *)cache)[at + d] = src[d];
                }
            }
        }
    }
    return ORACLE_OK;
}

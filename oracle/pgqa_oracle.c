/*
 * pgqa_oracle.c -- TEST INFRASTRUCTURE, not part of the library.
 *
 * A plain, slow CPU reference in fp64 for decode attention over a paged KV
 * cache with grouped-query heads, for the split-KV partial/merge identity it
 * rests on, and for the paged KV append.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg load this file.  It shares no code,
 * header, table or helper with the CUDA library; neither includes the other.
 *
 * What is computed, and where it is stated:
 *   - KV pool layout [pages, page_size, kv_heads, head_dim] and the append as
 *     one copy of each new token's row into its flat slot
 *     ("flashlet" README, design bullets: pool layout matches NHD, set_kv is a
 *     single index_copy_).
 *   - Page table in CSR form (kv_indptr, kv_indices, last_page_len) and one
 *     ragged call whose qo_indptr mixes a prefill chunk with decode rows under a
 *     causal mask ("flashlet" README, design bullets: ragged plan()/run()).
 *   - The attention itself is the plain definition the engines check against:
 *     softmax(q K^T * scale) V per head over the request's cached keys
 *     ("flashlet" README, layout: torch_backend.py is the dense SDPA
 *     correctness oracle; "A library kernel for decode", section "Why 18% of
 *     the outputs changed": the kernel is checked against plain attention on a
 *     rebuilt cache).
 *   - Split-KV: a request's keys are cut into slices, a partial result is
 *     computed per slice and the partials are merged ("A library kernel for
 *     decode", section "What changed").  The merge is the log-sum-exp identity
 *     written out below.
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *   - query head h reads kv head floor(h / g), g = Hq / Hkv (contiguous groups,
 *     the grouping of the Qwen2.5 models the pages run);
 *   - kv_len = (npages - 1) * page_size + last_page_len, 0 when npages == 0;
 *   - causal alignment is bottom-right: query row i of a segment of L rows over
 *     N keys may attend keys j <= N - L + i;
 *   - scale defaults to 1/sqrt(head_dim); lse is the natural log-sum-exp of the
 *     scaled scores; a row with no admissible key has o = 0 and lse = -inf;
 *   - a negative slot in the append means "skip this token";
 *   - RoPE, which the pages name but do not write out ("flashlet" README,
 *     milestones: a RoPE fusion kernel; "Torchlet", introduction: the
 *     Qwen2.5-style model includes RoPE), is read as the rotate-half form of the
 *     Qwen2.5 models: channel i < d/2 pairs with channel i + d/2 and both turn
 *     by the angle pos * theta^(-2i/d), theta a parameter; the rotated value is
 *     rounded once to the 16-bit type, to nearest with ties to even.
 *
 * Everything is fp64.  16-bit inputs are widened exactly (every bf16 and fp16
 * value is a double).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BF16 0
#define ORACLE_FP16 1

#define ORACLE_OK 0
#define ORACLE_ERR_PAGE_INDEX (-1)
#define ORACLE_ERR_LAST_PAGE_LEN (-2)
#define ORACLE_ERR_INDPTR (-3)
#define ORACLE_ERR_ARG (-4)
#define ORACLE_ERR_NOMEM (-5)

/* Exact widening of a 16-bit float pattern to double.
 * bf16: the upper half of an IEEE binary32.  fp16: IEEE binary16
 * (1 sign, 5 exponent bits with bias 15, 10 fraction bits). */
double oracle_widen(uint16_t bits, int dtype)
{
    if (dtype == ORACLE_BF16) {
        uint32_t u = (uint32_t)bits << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 31;
    int m = bits & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);             /* zero or subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* kv_len of request b from its page count and the fill of its last page. */
int64_t oracle_kv_len(const int32_t *kv_indptr, const int32_t *last_page_len,
                      int b, int page_size)
{
    int64_t npages = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    if (npages == 0)
        return 0;
    return (npages - 1) * page_size + last_page_len[b];
}

/* Checks the page table the way the method needs it: monotone indptr,
 * every page index inside the pool, last_page_len in [1, page_size] for a
 * request with pages and 0 for one without. */
int oracle_check_page_table(const int32_t *kv_indptr, const int32_t *kv_indices,
                            const int32_t *last_page_len, int batch,
                            int64_t num_pages, int page_size)
{
    if (kv_indptr[0] != 0)
        return ORACLE_ERR_INDPTR;
    for (int b = 0; b < batch; ++b) {
        if (kv_indptr[b + 1] < kv_indptr[b])
            return ORACLE_ERR_INDPTR;
        int64_t npages = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
        if (npages == 0 && last_page_len[b] != 0)
            return ORACLE_ERR_LAST_PAGE_LEN;
        if (npages > 0 && (last_page_len[b] < 1 || last_page_len[b] > page_size))
            return ORACLE_ERR_LAST_PAGE_LEN;
        for (int64_t i = kv_indptr[b]; i < kv_indptr[b + 1]; ++i)
            if (kv_indices[i] < 0 || kv_indices[i] >= num_pages)
                return ORACLE_ERR_PAGE_INDEX;
    }
    return ORACLE_OK;
}

/* Paged KV append: token t's rows k[t], v[t] ([Hkv, d] each, row_bytes bytes)
 * are copied to flat slot slot_mapping[t] of the pools viewed as
 * [pages * page_size, Hkv, d].  Byte copy, so bit-exact by construction. */
int oracle_kv_append(uint8_t *k_pool, uint8_t *v_pool, int64_t num_slots,
                     int64_t row_bytes, const uint8_t *k, const uint8_t *v,
                     const int64_t *slot_mapping, int64_t num_tokens)
{
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= num_slots)
            return ORACLE_ERR_PAGE_INDEX;
        memcpy(k_pool + s * row_bytes, k + t * row_bytes, (size_t)row_bytes);
        memcpy(v_pool + s * row_bytes, v + t * row_bytes, (size_t)row_bytes);
    }
    return ORACLE_OK;
}

/* Gathers the dense keys and values of request b, kv head kvh, as rows
 * 0..n-1: row j lives in page kv_indices[kv_indptr[b] + j / page_size] at
 * offset j % page_size. */
static void gather_dense(const uint16_t *k_pool, const uint16_t *v_pool, int dtype,
                         int page_size, int Hkv, int d, const int32_t *kv_indptr,
                         const int32_t *kv_indices, int b, int kvh, int64_t n,
                         double *K, double *V)
{
    for (int64_t j = 0; j < n; ++j) {
        int64_t page = kv_indices[kv_indptr[b] + j / page_size];
        int64_t off = j % page_size;
        int64_t base = ((page * page_size + off) * Hkv + kvh) * (int64_t)d;
        for (int c = 0; c < d; ++c) {
            K[j * d + c] = oracle_widen(k_pool[base + c], dtype);
            V[j * d + c] = oracle_widen(v_pool[base + c], dtype);
        }
    }
}

/* Plain attention of one query vector over dense keys/values rows [j0, j1):
 *   s_j = scale * (q . K_j),  m = max_j s_j,  w_j = exp(s_j - m),
 *   o = sum_j w_j V_j / sum_j w_j,  lse = m + log(sum_j w_j).
 * An empty range gives o = 0, lse = -inf (the neutral element of the merge). */
static int attend_range(const double *qv, const double *K, const double *V,
                        int64_t j0, int64_t j1, int d, double scale,
                        double *o, double *lse)
{
    for (int c = 0; c < d; ++c)
        o[c] = 0.0;
    if (j1 <= j0) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    double *w = (double *)malloc((size_t)(j1 - j0) * sizeof(double));
    if (!w)
        return ORACLE_ERR_NOMEM;
    double m = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += qv[c] * K[j * d + c];
        w[j - j0] = scale * dot;
        if (w[j - j0] > m)
            m = w[j - j0];
    }
    double z = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
        w[j - j0] = exp(w[j - j0] - m);
        z += w[j - j0];
    }
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t j = j0; j < j1; ++j)
            acc += w[j - j0] * V[j * d + c];
        o[c] = acc / z;
    }
    *lse = m + log(z);
    free(w);
    return ORACLE_OK;
}

/* Log-sum-exp merge of n partials (o_s, lse_s), each o_s normalised over its
 * own slice:  lse = log sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s.
 * Partials with lse_s = -inf (empty slices) carry no weight. */
void oracle_lse_merge(int n, int d, const double *o_parts, const double *lse_parts,
                      double *o, double *lse)
{
    double m = -INFINITY;
    for (int s = 0; s < n; ++s)
        if (lse_parts[s] > m)
            m = lse_parts[s];
    for (int c = 0; c < d; ++c)
        o[c] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int s = 0; s < n; ++s)
        if (lse_parts[s] != -INFINITY)
            z += exp(lse_parts[s] - m);
    for (int s = 0; s < n; ++s) {
        if (lse_parts[s] == -INFINITY)
            continue;
        double w = exp(lse_parts[s] - m) / z;
        for (int c = 0; c < d; ++c)
            o[c] += w * o_parts[(int64_t)s * d + c];
    }
    *lse = m + log(z);
}

/* Problem description shared by the entry points below. */
typedef struct {
    const uint16_t *q;      /* [rows, Hq, d] */
    const uint16_t *k_pool; /* [num_pages, page_size, Hkv, d] */
    const uint16_t *v_pool;
    int dtype;
    int64_t num_pages;
    int page_size, Hq, Hkv, d;
    const int32_t *kv_indptr, *kv_indices, *last_page_len;
    const int32_t *qo_indptr; /* NULL: request b owns exactly query row b */
    int batch;
    int causal;
    double scale;
    double *out; /* [rows, Hq, d] */
    double *lse; /* [rows, Hq] */
    /* work distribution */
    int nthreads;
    int err;
} problem_t;

typedef struct {
    problem_t *p;
    int tid;
} worker_t;

static int64_t q_begin(const problem_t *p, int b) { return p->qo_indptr ? p->qo_indptr[b] : b; }
static int64_t q_end(const problem_t *p, int b) { return p->qo_indptr ? p->qo_indptr[b + 1] : b + 1; }

/* One unit of work: request b, query head h (all of the request's rows). */
static int run_unit(problem_t *p, int b, int h)
{
    const int g = p->Hq / p->Hkv;
    const int kvh = h / g;
    const int d = p->d;
    int64_t n = oracle_kv_len(p->kv_indptr, p->last_page_len, b, p->page_size);
    int64_t r0 = q_begin(p, b), r1 = q_end(p, b), L = r1 - r0;
    double *K = (double *)malloc((size_t)(n > 0 ? n : 1) * d * sizeof(double));
    double *V = (double *)malloc((size_t)(n > 0 ? n : 1) * d * sizeof(double));
    double *qv = (double *)malloc((size_t)d * sizeof(double));
    if (!K || !V || !qv) {
        free(K); free(V); free(qv);
        return ORACLE_ERR_NOMEM;
    }
    gather_dense(p->k_pool, p->v_pool, p->dtype, p->page_size, p->Hkv, d,
                 p->kv_indptr, p->kv_indices, b, kvh, n, K, V);
    int rc = ORACLE_OK;
    for (int64_t r = r0; r < r1 && rc == ORACLE_OK; ++r) {
        int64_t i = r - r0;
        int64_t allowed = n;
        if (p->causal) {
            allowed = n - L + i + 1;
            if (allowed < 0) allowed = 0;
            if (allowed > n) allowed = n;
        }
        for (int c = 0; c < d; ++c)
            qv[c] = oracle_widen(p->q[(r * p->Hq + h) * (int64_t)d + c], p->dtype);
        rc = attend_range(qv, K, V, 0, allowed, d, p->scale,
                          p->out + (r * p->Hq + h) * (int64_t)d, p->lse + r * p->Hq + h);
    }
    free(K); free(V); free(qv);
    return rc;
}

static void *worker_main(void *arg)
{
    worker_t *w = (worker_t *)arg;
    problem_t *p = w->p;
    int64_t units = (int64_t)p->batch * p->Hq;
    for (int64_t u = w->tid; u < units; u += p->nthreads) {
        int rc = run_unit(p, (int)(u / p->Hq), (int)(u % p->Hq));
        if (rc != ORACLE_OK)
            p->err = rc; /* any non-zero value; races only between error codes */
    }
    return NULL;
}

/* Paged GQA attention for every query row of every request.
 * Returns ORACLE_OK, or a negative code for a malformed page table / argument.
 * nthreads <= 1 runs on the calling thread. */
int oracle_paged_attention(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                           int dtype, int64_t num_pages, int page_size, int Hq, int Hkv, int d,
                           const int32_t *kv_indptr, const int32_t *kv_indices,
                           const int32_t *last_page_len, const int32_t *qo_indptr, int batch,
                           int causal, double scale, double *out, double *lse, int nthreads)
{
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page_size <= 0 || batch < 0)
        return ORACLE_ERR_ARG;
    int rc = oracle_check_page_table(kv_indptr, kv_indices, last_page_len, batch,
                                     num_pages, page_size);
    if (rc != ORACLE_OK)
        return rc;
    if (scale <= 0.0)
        scale = 1.0 / sqrt((double)d);
    problem_t p = {q, k_pool, v_pool, dtype, num_pages, page_size, Hq, Hkv, d,
                   kv_indptr, kv_indices, last_page_len, qo_indptr, batch, causal, scale,
                   out, lse, nthreads < 1 ? 1 : nthreads, ORACLE_OK};
    if (p.nthreads == 1) {
        worker_t w = {&p, 0};
        worker_main(&w);
        return p.err;
    }
    pthread_t *th = (pthread_t *)malloc((size_t)p.nthreads * sizeof(pthread_t));
    worker_t *ws = (worker_t *)malloc((size_t)p.nthreads * sizeof(worker_t));
    if (!th || !ws) {
        free(th); free(ws);
        return ORACLE_ERR_NOMEM;
    }
    int started = 0;
    for (int t = 0; t < p.nthreads; ++t) {
        ws[t].p = &p;
        ws[t].tid = t;
        if (pthread_create(&th[t], NULL, worker_main, &ws[t]) != 0)
            break;
        ++started;
    }
    /* threads that failed to start leave their units to a serial sweep */
    for (int t = started; t < p.nthreads; ++t)
        worker_main(&ws[t]);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th); free(ws);
    return p.err;
}

/* Split-KV partial of one query row r, head h of request b over key slice
 * [j0, j1) (clipped to the causal bound of that row): o normalised over the
 * slice and lse of the slice, as in attend_range. */
int oracle_attention_partial(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                             int dtype, int page_size, int Hq, int Hkv, int d,
                             const int32_t *kv_indptr, const int32_t *kv_indices,
                             const int32_t *last_page_len, const int32_t *qo_indptr,
                             int b, int64_t r, int h, int64_t j0, int64_t j1, int causal,
                             double scale, double *o, double *lse)
{
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
        return ORACLE_ERR_ARG;
    if (scale <= 0.0)
        scale = 1.0 / sqrt((double)d);
    const int g = Hq / Hkv, kvh = h / g;
    int64_t n = oracle_kv_len(kv_indptr, last_page_len, b, page_size);
    int64_t r0 = qo_indptr ? qo_indptr[b] : b, r1 = qo_indptr ? qo_indptr[b + 1] : b + 1;
    int64_t allowed = n;
    if (causal) {
        allowed = n - (r1 - r0) + (r - r0) + 1;
        if (allowed < 0) allowed = 0;
        if (allowed > n) allowed = n;
    }
    if (j1 > allowed) j1 = allowed;
    if (j0 < 0) j0 = 0;
    double *K = (double *)malloc((size_t)(n > 0 ? n : 1) * d * sizeof(double));
    double *V = (double *)malloc((size_t)(n > 0 ? n : 1) * d * sizeof(double));
    double *qv = (double *)malloc((size_t)d * sizeof(double));
    if (!K || !V || !qv) {
        free(K); free(V); free(qv);
        return ORACLE_ERR_NOMEM;
    }
    gather_dense(k_pool, v_pool, dtype, page_size, Hkv, d, kv_indptr, kv_indices, b, kvh, n, K, V);
    for (int c = 0; c < d; ++c)
        qv[c] = oracle_widen(q[(r * Hq + h) * (int64_t)d + c], dtype);
    int rc = attend_range(qv, K, V, j0, j1, d, scale, o, lse);
    free(K); free(V); free(qv);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Narrowing and the rotary position embedding.                             */
/* ------------------------------------------------------------------------ */

/* Rounds x to the 16-bit type, to nearest with ties to even, straight from the
 * double (no binary32 step in between, which could round twice) and returns
 * the bit pattern.  bf16: 8 significant bits, exponents -126..127 (the range of
 * binary32); fp16: 11 significant bits, exponents -14..15.  Below the smallest
 * normal the spacing stays that of the smallest binade (subnormals); past the
 * largest finite value the result is infinity; NaN stays NaN. */
uint16_t oracle_narrow(double x, int dtype)
{
    const int bf = dtype == ORACLE_BF16;
    const int prec = bf ? 8 : 11;
    const int emin = bf ? -126 : -14, emax = bf ? 127 : 15;
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | (bf ? 0x7FC0u : 0x7E00u));
    const uint16_t inf = (uint16_t)(sign | (bf ? 0x7F80u : 0x7C00u));
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return inf;
    int ex;
    frexp(a, &ex);            /* a = f * 2^ex, f in [0.5, 1): binade exponent ex - 1 */
    int e = ex - 1;
    if (e < emin)
        e = emin;
    /* a in units of the spacing 2^(e - prec + 1): an integer part and an exact fraction */
    double y = ldexp(a, prec - 1 - e);
    double fl = floor(y), frac = y - fl;
    double r = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;
    /* r * 2^(e - prec + 1); r may have carried to 2^prec (the next binade) */
    int eb = e;
    if (r >= ldexp(1.0, prec)) {
        r = ldexp(r, -1);
        eb = e + 1;
    }
    if (eb > emax)
        return inf;
    uint32_t mant = (uint32_t)r;  /* prec bits when normal, fewer when subnormal */
    int normal = mant >= (1u << (prec - 1));
    uint32_t bits;
    if (bf) {
        int biased = normal ? eb + 127 : 0;
        bits = ((uint32_t)biased << 7) | (mant & 0x7Fu);
    } else {
        int biased = normal ? eb + 15 : 0;
        bits = ((uint32_t)biased << 10) | (mant & 0x3FFu);
    }
    return (uint16_t)(sign | bits);
}

/* Rotary position embedding in fp64 on rows [rows, heads, d] at positions[rows]:
 * for i < d/2, with phi = positions[r] * theta^(-2i/d),
 *     y[i]       = x[i] cos(phi) - x[i + d/2] sin(phi)
 *     y[i + d/2] = x[i + d/2] cos(phi) + x[i] sin(phi). */
int oracle_rope_f64(const double *x, double *y, int64_t rows, int heads, int d,
                    const int32_t *positions, double theta)
{
    if (rows < 0 || heads <= 0 || d <= 0 || d % 2 != 0 || !(theta > 0.0))
        return ORACLE_ERR_ARG;
    const int half = d / 2;
    for (int64_t r = 0; r < rows; ++r) {
        const double pos = (double)positions[r];
        for (int i = 0; i < half; ++i) {
            const double phi = pos * pow(theta, -2.0 * i / d);
            const double c = cos(phi), s = sin(phi);
            for (int h = 0; h < heads; ++h) {
                const int64_t base = (r * heads + h) * (int64_t)d;
                const double a = x[base + i], b = x[base + i + half];
                y[base + i] = a * c - b * s;
                y[base + i + half] = b * c + a * s;
            }
        }
    }
    return ORACLE_OK;
}

/* The same on 16-bit patterns: widened exactly, rotated in fp64, then (out16)
 * narrowed once; out64 (optional) receives the fp64 values before rounding. */
int oracle_rope(const uint16_t *x, int64_t rows, int heads, int d, const int32_t *positions,
                double theta, int dtype, double *out64, uint16_t *out16)
{
    if (rows < 0 || heads <= 0 || d <= 0)
        return ORACLE_ERR_ARG;
    const int64_t n = rows * heads * (int64_t)d;
    if (n == 0)
        return ORACLE_OK;
    double *xin = (double *)malloc((size_t)n * sizeof(double));
    double *y = (double *)malloc((size_t)n * sizeof(double));
    if (!xin || !y) {
        free(xin); free(y);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t k = 0; k < n; ++k)
        xin[k] = oracle_widen(x[k], dtype);
    int rc = oracle_rope_f64(xin, y, rows, heads, d, positions, theta);
    if (rc == ORACLE_OK) {
        for (int64_t k = 0; k < n; ++k) {
            if (out64) out64[k] = y[k];
            if (out16) out16[k] = oracle_narrow(y[k], dtype);
        }
    }
    free(xin); free(y);
    return rc;
}

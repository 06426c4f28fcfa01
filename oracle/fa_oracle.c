/*
 * CPU FP64 oracle for exact attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It shares no code, header or constant with the CUDA
 * path, and it is deliberately plain and slow: every query row materialises
 * its full score row S[i, :], runs the three-pass safe softmax and then forms
 * P @ V, exactly as the definition reads.  No blocking, no fusion.
 *
 * Sources (page titles, then the section / function on the page):
 *   [flash_lab]  "flash_lab.py -- FlashAttention, flash-decoding and
 *                megakernel in numpy" (CS349E lecture 11 shared module):
 *                module docstring (conventions: Q[N,d], K[Nk,d], V[Nk,dv],
 *                scale 1/sqrt(d), query i at position Nk-N+i),
 *                section 1 `softmax_3pass`, section 2 `_causal_mask` and
 *                `standard_attention`, section 3 `flash_fwd` (L = m + log l),
 *                section 4 `split_kv_decode` (lse merge).
 *                section 2 `standard_attention_bwd` (dV = P^T dO, dP = dO V^T,
 *                dS = P o (dP - D) with D_i = sum dO_i o O_i, dQ = dS K scale,
 *                dK = dS^T Q scale).
 *   [fwd_demo]   "02_flash_forward.py -- FlashAttention forward" (CS349E
 *                lecture 11), demo 1: causal position convention for N != Nk.
 *
 * Readings where the pages are silent or disagree:
 *   - A query row with no visible key (only possible when causal and N > Nk):
 *     the pages give NaN (`standard_attention`), O = 0 (`flash_fwd` order
 *     fa1) or weight 0 for an all -inf segment (`merge_states`).  This oracle
 *     writes O = 0 and LSE = -inf for such a row.
 *   - LSE is the natural logarithm of sum_j exp(scale * q.k_j) over visible
 *     keys, i.e. it includes the scale ([flash_lab] section 3, L = m + log l).
 *
 * Inputs are either float64 arrays or bf16 bit patterns (uint16); a bf16
 * value is widened exactly (its 16 bits become the top half of a float32,
 * which converts exactly to float64).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

/* ---------------------------------------------------------------------- */
/* exact bf16 -> double widening                                           */
/* ---------------------------------------------------------------------- */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static void widen_bf16(const uint16_t* src, double* dst, long n)
{
    for (long i = 0; i < n; ++i) dst[i] = bf16_to_double(src[i]);
}

/* ---------------------------------------------------------------------- */
/* one query row of standard attention                                     */
/* ---------------------------------------------------------------------- */
/*
 * [flash_lab] section 2 `standard_attention` for a single query row i:
 *   S[i, j] = scale * sum_c Q[i, c] K[j, c]                 (score row)
 *   masked to -inf where key position j > query position (causal,
 *   [flash_lab] `_causal_mask` with offset Nk - N)
 *   P[i, :] = softmax_3pass(S[i, :])  -- pass 1 max, pass 2 sum of exp,
 *             pass 3 divide ([flash_lab] section 1 `softmax_3pass`)
 *   O[i, :] = sum_j P[i, j] V[j, :]
 *   LSE[i]  = m + log(sum_j exp(S[i, j] - m))
 * `qpos` is the query's position (Nk - N + i); pass LONG_MAX-like values
 * (>= Nk - 1) for a non-causal row.  `s` is caller scratch of length Nk.
 */
static void attention_row(const double* q, const double* K, const double* V, long Nk, long d,
                          long dv, long qpos, double scale, double* s, double* o, double* lse)
{
    /* S row, with the causal mask applied as -inf */
    for (long j = 0; j < Nk; ++j) {
        if (j > qpos) {
            s[j] = -INFINITY;
            continue;
        }
        const double* k = K + j * d;
        double acc = 0.0;
        for (long c = 0; c < d; ++c) acc += q[c] * k[c];
        s[j] = acc * scale;
    }
    /* pass 1: row max */
    double m = -INFINITY;
    for (long j = 0; j < Nk; ++j)
        if (s[j] > m) m = s[j];
    for (long c = 0; c < dv; ++c) o[c] = 0.0;
    if (m == -INFINITY) { /* no visible key: O = 0, LSE = -inf (reading above) */
        *lse = -INFINITY;
        return;
    }
    /* pass 2: sum of exp(S - m) */
    double l = 0.0;
    for (long j = 0; j < Nk; ++j) {
        s[j] = exp(s[j] - m); /* exp(-inf) = 0 for masked keys */
        l += s[j];
    }
    /* pass 3: divide, then P @ V */
    for (long j = 0; j < Nk; ++j) {
        double p = s[j] / l;
        if (p == 0.0) continue;
        const double* v = V + j * dv;
        for (long c = 0; c < dv; ++c) o[c] += p * v[c];
    }
    *lse = m + log(l);
}

/* ---------------------------------------------------------------------- */
/* thread pool over work items                                              */
/* ---------------------------------------------------------------------- */
typedef struct {
    /* shared description of the batch */
    const void* Q;
    const void* K;
    const void* V;
    int bf16; /* inputs are bf16 bits (1) or float64 (0) */
    long BH, N, Nk, d, dv;
    long q_stride_bh, k_stride_bh, v_stride_bh; /* elements between heads */
    const int* seqlens;                         /* decode only: length per batch index */
    long H;                                     /* decode only */
    int causal;
    double scale;
    long row0, row1, chunk;
    double* O;
    double* LSE;
    /* scheduling */
    long n_items;
    long next;
    pthread_mutex_t lock;
    int failed;
} job_t;

static long take_item(job_t* jb)
{
    pthread_mutex_lock(&jb->lock);
    long it = jb->next < jb->n_items ? jb->next++ : -1;
    pthread_mutex_unlock(&jb->lock);
    return it;
}

/* Fetch `n` values at element offset `off` of input `src` as float64. */
static const double* fetch(const job_t* jb, const void* src, long off, long n, double* buf)
{
    if (jb->bf16) {
        widen_bf16((const uint16_t*)src + off, buf, n);
        return buf;
    }
    return (const double*)src + off;
}

static void* attention_worker(void* arg)
{
    job_t* jb = (job_t*)arg;
    long nrows = jb->row1 - jb->row0;
    long per_head = (nrows + jb->chunk - 1) / jb->chunk;
    double* s = malloc(sizeof(double) * (size_t)(jb->Nk > 0 ? jb->Nk : 1));
    double* qb = malloc(sizeof(double) * (size_t)jb->d);
    double* kb = jb->bf16 ? malloc(sizeof(double) * (size_t)(jb->Nk * jb->d + 1)) : NULL;
    double* vb = jb->bf16 ? malloc(sizeof(double) * (size_t)(jb->Nk * jb->dv + 1)) : NULL;
    if (!s || !qb || (jb->bf16 && (!kb || !vb))) {
        pthread_mutex_lock(&jb->lock);
        jb->failed = 1;
        pthread_mutex_unlock(&jb->lock);
        free(s); free(qb); free(kb); free(vb);
        return NULL;
    }
    long it;
    while ((it = take_item(jb)) >= 0) {
        long bh = it / per_head;
        long r0 = jb->row0 + (it % per_head) * jb->chunk;
        long r1 = r0 + jb->chunk < jb->row1 ? r0 + jb->chunk : jb->row1;
        const double* K = fetch(jb, jb->K, bh * jb->k_stride_bh, jb->Nk * jb->d, kb);
        const double* V = fetch(jb, jb->V, bh * jb->v_stride_bh, jb->Nk * jb->dv, vb);
        for (long i = r0; i < r1; ++i) {
            const double* q = jb->bf16
                ? fetch(jb, jb->Q, bh * jb->q_stride_bh + i * jb->d, jb->d, qb)
                : (const double*)jb->Q + bh * jb->q_stride_bh + i * jb->d;
            /* query i sits at position Nk - N + i ([fwd_demo] demo 1) */
            long qpos = jb->causal ? jb->Nk - jb->N + i : jb->Nk;
            long out = bh * nrows + (i - jb->row0);
            attention_row(q, K, V, jb->Nk, jb->d, jb->dv, qpos, jb->scale, s, jb->O + out * jb->dv,
                          jb->LSE + out);
        }
    }
    free(s); free(qb); free(kb); free(vb);
    return NULL;
}

static int run_pool(job_t* jb, void* (*fn)(void*), int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (jb->n_items < nthreads) nthreads = jb->n_items > 0 ? (int)jb->n_items : 1;
    pthread_t th[256];
    pthread_mutex_init(&jb->lock, NULL);
    jb->next = 0;
    jb->failed = 0;
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, fn, jb) != 0) break;
        ++started;
    }
    fn(jb); /* the calling thread works too */
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&jb->lock);
    return jb->failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* public entry points                                                      */
/* ---------------------------------------------------------------------- */
/*
 * Standard attention over BH independent heads ([flash_lab] section 2).
 * Q [BH,N,d], K [BH,Nk,d], V [BH,Nk,dv], either float64 (bf16 = 0) or bf16
 * bit patterns (bf16 = 1).  Only query rows [row0, row1) are computed;
 * O [BH, row1-row0, dv] and LSE [BH, row1-row0] are float64.
 */
int oracle_attention(const void* Q, const void* K, const void* V, int bf16, long BH, long N, long Nk,
                     long d, long dv, int causal, double scale, long row0, long row1, double* O,
                     double* LSE, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE || BH < 0 || N < 0 || Nk < 0 || d <= 0 || dv <= 0 ||
        row0 < 0 || row1 < row0 || row1 > N)
        return ORACLE_ERR_ARG;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.Q = Q; jb.K = K; jb.V = V; jb.bf16 = bf16;
    jb.BH = BH; jb.N = N; jb.Nk = Nk; jb.d = d; jb.dv = dv;
    jb.q_stride_bh = N * d; jb.k_stride_bh = Nk * d; jb.v_stride_bh = Nk * dv;
    jb.causal = causal; jb.scale = scale;
    jb.row0 = row0; jb.row1 = row1; jb.chunk = 64;
    jb.O = O; jb.LSE = LSE;
    long nrows = row1 - row0;
    jb.n_items = nrows > 0 ? BH * ((nrows + jb.chunk - 1) / jb.chunk) : 0;
    if (jb.n_items == 0) return ORACLE_OK;
    return run_pool(&jb, attention_worker, nthreads);
}

static void* decode_worker(void* arg)
{
    job_t* jb = (job_t*)arg;
    double* s = malloc(sizeof(double) * (size_t)(jb->Nk > 0 ? jb->Nk : 1));
    double* qb = malloc(sizeof(double) * (size_t)jb->d);
    double* kb = jb->bf16 ? malloc(sizeof(double) * (size_t)(jb->Nk * jb->d + 1)) : NULL;
    double* vb = jb->bf16 ? malloc(sizeof(double) * (size_t)(jb->Nk * jb->dv + 1)) : NULL;
    if (!s || !qb || (jb->bf16 && (!kb || !vb))) {
        pthread_mutex_lock(&jb->lock);
        jb->failed = 1;
        pthread_mutex_unlock(&jb->lock);
        free(s); free(qb); free(kb); free(vb);
        return NULL;
    }
    long bh;
    while ((bh = take_item(jb)) >= 0) {
        long b = bh / jb->H;
        long n = jb->seqlens[b];
        const double* q = fetch(jb, jb->Q, bh * jb->d, jb->d, qb);
        const double* K = fetch(jb, jb->K, bh * jb->k_stride_bh, n * jb->d, kb);
        const double* V = fetch(jb, jb->V, bh * jb->v_stride_bh, n * jb->dv, vb);
        /* a single query at position n - 1 sees all n cached keys */
        attention_row(q, K, V, n, jb->d, jb->dv, n, jb->scale, s, jb->O + bh * jb->dv,
                      jb->LSE + bh);
    }
    free(s); free(qb); free(kb); free(vb);
    return NULL;
}

/*
 * Single-query decode: for every (b, h), standard attention of q[b,h] over
 * the first seqlens[b] rows of the caches (no split; the split-and-merge of
 * [flash_lab] section 4 reaches this same value).  q [B*H, d],
 * K [B*H, Nk_max, d], V [B*H, Nk_max, dv]; O [B*H, dv], LSE [B*H] float64.
 */
int oracle_decode(const void* q, const void* K, const void* V, int bf16, const int* seqlens, long B,
                  long H, long Nk_max, long d, long dv, double scale, double* O, double* LSE,
                  int nthreads)
{
    if (!q || !K || !V || !seqlens || !O || !LSE || B < 0 || H < 0 || Nk_max < 0 || d <= 0 ||
        dv <= 0)
        return ORACLE_ERR_ARG;
    for (long b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > Nk_max) return ORACLE_ERR_ARG;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.Q = q; jb.K = K; jb.V = V; jb.bf16 = bf16;
    jb.Nk = Nk_max; jb.d = d; jb.dv = dv; jb.H = H;
    jb.k_stride_bh = Nk_max * d; jb.v_stride_bh = Nk_max * dv;
    jb.seqlens = seqlens; jb.scale = scale;
    jb.O = O; jb.LSE = LSE;
    jb.n_items = B * H;
    if (jb.n_items == 0) return ORACLE_OK;
    return run_pool(&jb, decode_worker, nthreads);
}

/*
 * Combine of split states in the log-sum-exp form ([flash_lab] section 4,
 * `split_kv_decode`): for each row,
 *   lse = log sum_s exp(lse_s)       (computed as M + log sum_s exp(lse_s - M),
 *                                     M = max_s lse_s)
 *   o   = sum_s exp(lse_s - lse) * o_s
 * A state with lse_s = -inf is an empty split and gets weight 0; if every
 * state of a row is empty the row is O = 0, LSE = -inf.
 * o_parts [P, rows, dv], lse_parts [P, rows]; o [rows, dv], lse [rows].
 */
int oracle_merge_lse(const double* o_parts, const double* lse_parts, long P, long rows, long dv,
                     double* o, double* lse)
{
    if (!o_parts || !lse_parts || !o || !lse || P < 0 || rows < 0 || dv <= 0) return ORACLE_ERR_ARG;
    for (long r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (long p = 0; p < P; ++p)
            if (lse_parts[p * rows + r] > M) M = lse_parts[p * rows + r];
        double* orow = o + r * dv;
        for (long c = 0; c < dv; ++c) orow[c] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (long p = 0; p < P; ++p) {
            double x = lse_parts[p * rows + r];
            if (x != -INFINITY) sum += exp(x - M);
        }
        double L = M + log(sum);
        lse[r] = L;
        for (long p = 0; p < P; ++p) {
            double x = lse_parts[p * rows + r];
            if (x == -INFINITY) continue;
            double w = exp(x - L);
            const double* op = o_parts + (p * rows + r) * dv;
            for (long c = 0; c < dv; ++c) orow[c] += w * op[c];
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* backward of standard attention                                          */
/* ---------------------------------------------------------------------- */
typedef struct {
    const void *Q, *K, *V, *dO;
    int bf16;
    long BH, N, Nk, d, dv;
    int causal;
    double scale;
    double *dQ, *dK, *dV;
    long next;
    pthread_mutex_t lock;
    int failed;
} bwd_job_t;

static long bwd_take(bwd_job_t* jb)
{
    pthread_mutex_lock(&jb->lock);
    long it = jb->next < jb->BH ? jb->next++ : -1;
    pthread_mutex_unlock(&jb->lock);
    return it;
}

static const double* bwd_fetch(const bwd_job_t* jb, const void* src, long off, long n, double* buf)
{
    if (jb->bf16) {
        widen_bf16((const uint16_t*)src + off, buf, n);
        return buf;
    }
    return (const double*)src + off;
}

/*
 * One head of [flash_lab] section 2 `standard_attention_bwd`, one query row
 * at a time.  For row i:
 *   P[i, :] from the forward definition (masked scores, 3-pass softmax);
 *   O[i, :]  = sum_j P[i, j] V[j, :]
 *   D[i]     = sum_c dO[i, c] O[i, c]
 *   dP[i, j] = sum_c dO[i, c] V[j, c]
 *   dS[i, j] = P[i, j] (dP[i, j] - D[i])
 *   dQ[i, :] = scale sum_j dS[i, j] K[j, :]
 *   dK[j, :] += scale dS[i, j] Q[i, :]      (summed over all rows i)
 *   dV[j, :] += P[i, j] dO[i, :]            (summed over all rows i)
 * A row with no visible key has a zero P row and contributes nothing.
 */
static void bwd_head(const double* Q, const double* K, const double* V, const double* dO, long N, long Nk,
                     long d, long dv, int causal, double scale, double* p, double* orow, double* dQ,
                     double* dK, double* dV)
{
    for (long j = 0; j < Nk * d; ++j) dK[j] = 0.0;
    for (long j = 0; j < Nk * dv; ++j) dV[j] = 0.0;
    for (long i = 0; i < N; ++i) {
        const double* q = Q + i * d;
        const double* g = dO + i * dv;
        double* dq = dQ + i * d;
        for (long c = 0; c < d; ++c) dq[c] = 0.0;
        long qpos = causal ? Nk - N + i : Nk; /* [fwd_demo] demo 1 */
        /* scores, masked */
        for (long j = 0; j < Nk; ++j) {
            if (j > qpos) {
                p[j] = -INFINITY;
                continue;
            }
            double acc = 0.0;
            for (long c = 0; c < d; ++c) acc += q[c] * K[j * d + c];
            p[j] = acc * scale;
        }
        /* 3-pass softmax: max, sum of exp, divide */
        double m = -INFINITY;
        for (long j = 0; j < Nk; ++j)
            if (p[j] > m) m = p[j];
        if (m == -INFINITY) continue; /* no visible key */
        double l = 0.0;
        for (long j = 0; j < Nk; ++j) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        for (long j = 0; j < Nk; ++j) p[j] /= l;
        /* O row and D */
        for (long c = 0; c < dv; ++c) orow[c] = 0.0;
        for (long j = 0; j < Nk; ++j)
            for (long c = 0; c < dv; ++c) orow[c] += p[j] * V[j * dv + c];
        double D = 0.0;
        for (long c = 0; c < dv; ++c) D += g[c] * orow[c];
        /* dP, dS and the three products */
        for (long j = 0; j < Nk; ++j) {
            if (j > qpos) continue; /* masked key: P = 0 and dS = 0 */
            double dp = 0.0;
            for (long c = 0; c < dv; ++c) dp += g[c] * V[j * dv + c];
            double ds = p[j] * (dp - D);
            for (long c = 0; c < d; ++c) dq[c] += scale * ds * K[j * d + c];
            for (long c = 0; c < d; ++c) dK[j * d + c] += scale * ds * q[c];
            for (long c = 0; c < dv; ++c) dV[j * dv + c] += p[j] * g[c];
        }
    }
}

static void* bwd_worker(void* arg)
{
    bwd_job_t* jb = (bwd_job_t*)arg;
    long nq = jb->N * jb->d, nk = jb->Nk * jb->d, nv = jb->Nk * jb->dv, ng = jb->N * jb->dv;
    double* p = malloc(sizeof(double) * (size_t)(jb->Nk + 1));
    double* orow = malloc(sizeof(double) * (size_t)jb->dv);
    double* buf = jb->bf16 ? malloc(sizeof(double) * (size_t)(nq + nk + nv + ng + 1)) : NULL;
    if (!p || !orow || (jb->bf16 && !buf)) {
        pthread_mutex_lock(&jb->lock);
        jb->failed = 1;
        pthread_mutex_unlock(&jb->lock);
        free(p); free(orow); free(buf);
        return NULL;
    }
    long bh;
    while ((bh = bwd_take(jb)) >= 0) {
        const double* Q = bwd_fetch(jb, jb->Q, bh * nq, nq, buf);
        const double* K = bwd_fetch(jb, jb->K, bh * nk, nk, buf ? buf + nq : NULL);
        const double* V = bwd_fetch(jb, jb->V, bh * nv, nv, buf ? buf + nq + nk : NULL);
        const double* G = bwd_fetch(jb, jb->dO, bh * ng, ng, buf ? buf + nq + nk + nv : NULL);
        bwd_head(Q, K, V, G, jb->N, jb->Nk, jb->d, jb->dv, jb->causal, jb->scale, p, orow,
                 jb->dQ + bh * nq, jb->dK + bh * nk, jb->dV + bh * nv);
    }
    free(p); free(orow); free(buf);
    return NULL;
}

/*
 * Gradients of standard attention over BH independent heads for the upstream
 * gradient dO ([flash_lab] section 2 `standard_attention_bwd`).  Q [BH,N,d],
 * K [BH,Nk,d], V [BH,Nk,dv], dO [BH,N,dv], all float64 (bf16 = 0) or all bf16
 * bit patterns (bf16 = 1).  dQ [BH,N,d], dK [BH,Nk,d], dV [BH,Nk,dv] float64.
 * One head per work item; heads run on `nthreads` threads.
 */
int oracle_attention_bwd(const void* Q, const void* K, const void* V, const void* dO, int bf16, long BH,
                         long N, long Nk, long d, long dv, int causal, double scale, double* dQ,
                         double* dK, double* dV, int nthreads)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV || BH < 0 || N < 0 || Nk < 0 || d <= 0 || dv <= 0)
        return ORACLE_ERR_ARG;
    if (BH == 0) return ORACLE_OK;
    bwd_job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.Q = Q; jb.K = K; jb.V = V; jb.dO = dO; jb.bf16 = bf16;
    jb.BH = BH; jb.N = N; jb.Nk = Nk; jb.d = d; jb.dv = dv;
    jb.causal = causal; jb.scale = scale;
    jb.dQ = dQ; jb.dK = dK; jb.dV = dV;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (BH < nthreads) nthreads = (int)BH;
    pthread_t th[256];
    pthread_mutex_init(&jb.lock, NULL);
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, bwd_worker, &jb) != 0) break;
        ++started;
    }
    bwd_worker(&jb);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&jb.lock);
    return jb.failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * attn_oracle.c -- plain fp64 CPU attention forward: the ORACLE.
 *
 * This file is test infrastructure. Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark load it; the CUDA library never does, and
 * this file includes nothing from it.
 *
 * What it computes (for every batch b, head h and query row i):
 *
 *   t_j   = scale * sum_c q_ic * k_jc                  (fp64, exact bf16 inputs)
 *   valid = { j in [0, N_kv) : !causal || j <= i + off }
 *   valid empty  ->  O_i = 0, LSE_i = -inf
 *   otherwise       m = max_{j in valid} t_j
 *                   l = sum_{j in valid} exp(t_j - m)
 *                   O_i = sum_{j in valid} exp(t_j - m) * v_j / l
 *                   LSE_i = m + ln(l)
 *
 * Sources (the method reaches exactly this result, up to rounding order):
 *  - "Flash Attention 4" (mlc.ai, Modern GPU Programming for MLSys), section
 *    "算法结构" (algorithm structure): the definitions of p_ij, l_i, o_i and
 *    O_i = o_i / l_i, and the statement that the blocked method returns the same
 *    result as standard attention (overview).
 *  - same page, section "重缩放与结果写回" (rescale and write-back): LSE is the
 *    natural log of the row sum plus the reference times the scale, and rows
 *    with no valid key have LSE = -inf; the pseudo-code in "算法结构" stores 0
 *    for rows whose row_sum is 0.
 *  - same page, section "Causal Mask": the bottom-right aligned mask, query i
 *    sees keys j <= i + N_kv - N_q, capped at N_kv - 1 (off = N_kv - N_q).
 *    With off = 0 and N_q != N_kv the same code gives the top-left mask of
 *    "FlashAttention：一次前向计算" (qingsen), section on causal masking, fig. 12.
 *  - "FlashAttention：一次前向计算", section "先看 attention 最后要得到什么":
 *    S = QK^T, P = softmax_row(s*S), O = PV, with an explicit scale s.
 *  - "Flash Attention 4", section "GQA 支持" (grouped-query attention): with
 *    H query heads and H_kv key/value heads (H a multiple of H_kv), query head h
 *    reads key/value head h / (H / H_kv): the group of H / H_kv consecutive
 *    query heads kv*G .. kv*G + G - 1 shares K/V head kv. H_kv = H is plain
 *    multi-head attention.
 *  - Element types: inputs are bf16 or IEEE fp16 bit patterns ("Flash
 *    Attention 4", section "编译与验证", runs the kernel on fp16 tensors);
 *    each is widened exactly to double before any arithmetic.
 *
 * The computation is two passes per row (max, then the exponentials and the
 * weighted sum of V); no blocking, no delayed rescaling, no reordering. Work
 * is split over (b, h, block of rows) between POSIX threads, which changes
 * nothing in any row's arithmetic.
 *
 * Layouts (row-major, elements):
 *   fixed length:  q [B, Nq, H, d], k and v [B, Nkv, H_kv, d]  (16-bit patterns)
 *                  o [B, Nq, H, d] (double), lse [B, H, Nq] (double)
 *   varlen:        q [T, H, d], k and v [T, H_kv, d] packed by cu_seqlens
 *                  o [T, H, d] (double), lse [H, T] (double)
 * dtype: ORACLE_BF16 (0) or ORACLE_F16 (1), the type of all of q, k, v.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_BF16 = 0, ORACLE_F16 = 1 };

/* bf16 is the upper half of an IEEE binary32 word. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Subnormals are fraction * 2^-24; normal numbers (1024 + fraction) * 2^(e-25). */
static double f16_to_double(uint16_t h)
{
    const int sign = h >> 15, e = (h >> 10) & 31, f = h & 1023;
    double x;
    if (e == 0) x = ldexp((double)f, -24);
    else if (e == 31) x = f ? NAN : INFINITY;
    else x = ldexp((double)(1024 + f), e - 25);
    return sign ? -x : x;
}

static double to_double(uint16_t h, int dtype)
{
    return dtype == ORACLE_F16 ? f16_to_double(h) : bf16_to_double(h);
}

/* One query row against the key/value rows [0, nvalid) of one head.
 * k_rows / v_rows: double [nkv_rows, d] contiguous; t: scratch [nvalid]. */
static void attend_row(const double *q, const double *k_rows, const double *v_rows,
                       int64_t nvalid, int64_t d, double scale, double *t,
                       double *o, double *lse)
{
    int64_t j, c;
    if (nvalid <= 0) {
        for (c = 0; c < d; ++c) o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (j = 0; j < nvalid; ++j) {
        const double *kj = k_rows + j * d;
        double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
        for (c = 0; c + 3 < d; c += 4) {
            a0 += q[c] * kj[c];
            a1 += q[c + 1] * kj[c + 1];
            a2 += q[c + 2] * kj[c + 2];
            a3 += q[c + 3] * kj[c + 3];
        }
        for (; c < d; ++c) a0 += q[c] * kj[c];
        t[j] = scale * ((a0 + a1) + (a2 + a3));
        if (t[j] > m) m = t[j];
    }
    double l = 0.0;
    for (c = 0; c < d; ++c) o[c] = 0.0;
    for (j = 0; j < nvalid; ++j) {
        double p = exp(t[j] - m);
        const double *vj = v_rows + j * d;
        l += p;
        for (c = 0; c < d; ++c) o[c] += p * vj[c];
    }
    for (c = 0; c < d; ++c) o[c] /= l;
    *lse = m + log(l);
}

/* Number of valid keys for query row i (prefix [0, n)). */
static int64_t valid_keys(int64_t i, int64_t nkv, int causal, int64_t off)
{
    if (!causal) return nkv;
    int64_t n = i + off + 1;
    if (n < 0) n = 0;
    if (n > nkv) n = nkv;
    return n;
}

/* ------------------------------------------------------------------------ */
/* A "head problem" is one (sequence, head): rows of Q, K, V addressed by a
 * base pointer and a row stride (elements).                                 */
typedef struct {
    const uint16_t *q, *k, *v;   /* first row of this head (k, v: its K/V head) */
    int64_t row_stride;          /* elements between consecutive q / o rows  */
    int64_t kv_row_stride;       /* elements between consecutive k / v rows */
    int64_t nq, nkv, off;
    double *o;                   /* first output row (same stride as q)      */
    double *lse;                 /* lse of row 0; rows are contiguous        */
    int64_t row_begin, row_end;  /* rows of this work item                   */
} work_item;

typedef struct {
    const work_item *items;
    int64_t n_items;
    int64_t d;
    double scale;
    int causal;
    int dtype;
    int64_t next;                /* atomic work counter                      */
    int failed;
} pool_t;

static void run_item(const work_item *w, int64_t d, double scale, int causal, int dtype,
                     int *failed)
{
    int64_t i, c, j;
    /* keys needed by the last row of the item */
    int64_t need = 0;
    for (i = w->row_begin; i < w->row_end; ++i) {
        int64_t n = valid_keys(i, w->nkv, causal, w->off);
        if (n > need) need = n;
    }
    double *kd = (double *)malloc(sizeof(double) * (size_t)((need > 0 ? need : 1) * d));
    double *vd = (double *)malloc(sizeof(double) * (size_t)((need > 0 ? need : 1) * d));
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);
    double *t = (double *)malloc(sizeof(double) * (size_t)(need > 0 ? need : 1));
    if (!kd || !vd || !qd || !t) {
        __atomic_store_n(failed, 1, __ATOMIC_RELAXED);
        free(kd); free(vd); free(qd); free(t);
        return;
    }
    for (j = 0; j < need; ++j)
        for (c = 0; c < d; ++c) {
            kd[j * d + c] = to_double(w->k[j * w->kv_row_stride + c], dtype);
            vd[j * d + c] = to_double(w->v[j * w->kv_row_stride + c], dtype);
        }
    for (i = w->row_begin; i < w->row_end; ++i) {
        for (c = 0; c < d; ++c) qd[c] = to_double(w->q[i * w->row_stride + c], dtype);
        attend_row(qd, kd, vd, valid_keys(i, w->nkv, causal, w->off), d, scale, t,
                   w->o + i * w->row_stride, w->lse + i);
    }
    free(kd); free(vd); free(qd); free(t);
}

static void *pool_worker(void *arg)
{
    pool_t *p = (pool_t *)arg;
    for (;;) {
        int64_t idx = __atomic_fetch_add(&p->next, 1, __ATOMIC_RELAXED);
        if (idx >= p->n_items) break;
        run_item(&p->items[idx], p->d, p->scale, p->causal, p->dtype, &p->failed);
    }
    return NULL;
}

static int run_pool(const work_item *items, int64_t n_items, int64_t d, double scale,
                    int causal, int dtype, int nthreads)
{
    pool_t p;
    p.items = items; p.n_items = n_items; p.d = d; p.scale = scale;
    p.causal = causal; p.dtype = dtype; p.next = 0; p.failed = 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if ((int64_t)nthreads > n_items) nthreads = (int)(n_items > 0 ? n_items : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -2;
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, pool_worker, &p) != 0) break;
        ++started;
    }
    pool_worker(&p);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    free(th);
    return p.failed ? -2 : 0;
}

#define ROWS_PER_ITEM 64

/* Valid head counts and element type. */
static int heads_ok(int64_t H, int64_t Hkv, int dtype)
{
    return H >= 0 && Hkv >= 1 && (H == 0 || H % Hkv == 0) &&
           (dtype == ORACLE_BF16 || dtype == ORACLE_F16);
}

/* Fixed-length batch. Returns 0 on success, -1 on bad arguments, -2 on
 * allocation failure. off = Nkv - Nq gives the bottom-right aligned mask. */
int oracle_attention_bshd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t B, int64_t H, int64_t Hkv, int64_t Nq, int64_t Nkv, int64_t d,
                          int dtype, double scale, int causal, int64_t off,
                          double *o, double *lse, int nthreads)
{
    if (!q || !k || !v || !o || !lse || B < 0 || !heads_ok(H, Hkv, dtype) || Nq < 0 ||
        Nkv < 0 || d <= 0)
        return -1;
    const int64_t G = H > 0 ? H / Hkv : 1;
    int64_t chunks = (Nq + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM;
    int64_t n_items = B * H * chunks;
    if (n_items == 0) return 0;
    work_item *items = (work_item *)malloc(sizeof(work_item) * (size_t)n_items);
    if (!items) return -2;
    int64_t n = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t ch = 0; ch < chunks; ++ch) {
                work_item *w = &items[n++];
                w->q = q + (b * Nq * H + h) * d;
                w->k = k + (b * Nkv * Hkv + h / G) * d;
                w->v = v + (b * Nkv * Hkv + h / G) * d;
                w->row_stride = H * d;
                w->kv_row_stride = Hkv * d;
                w->nq = Nq; w->nkv = Nkv; w->off = off;
                w->o = o + (b * Nq * H + h) * d;
                w->lse = lse + (b * H + h) * Nq;
                w->row_begin = ch * ROWS_PER_ITEM;
                w->row_end = w->row_begin + ROWS_PER_ITEM < Nq ? w->row_begin + ROWS_PER_ITEM : Nq;
            }
    int rc = run_pool(items, n_items, d, scale, causal, dtype, nthreads);
    free(items);
    return rc;
}

/* Packed variable-length batch: sequence s owns rows [cu[s], cu[s+1]) of q, k, v
 * (self-attention, N_q = N_kv = length, so off = 0). lse is [H, T]. */
int oracle_attention_varlen(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const int32_t *cu_seqlens, int64_t num_seqs,
                            int64_t H, int64_t Hkv, int64_t d, int dtype, double scale, int causal,
                            double *o, double *lse, int nthreads)
{
    if (!q || !k || !v || !o || !lse || !cu_seqlens || num_seqs < 0 || !heads_ok(H, Hkv, dtype) ||
        d <= 0)
        return -1;
    const int64_t G = H > 0 ? H / Hkv : 1;
    if (cu_seqlens[0] != 0) return -1;
    int64_t T = cu_seqlens[num_seqs];
    int64_t n_items = 0;
    for (int64_t s = 0; s < num_seqs; ++s) {
        int64_t L = (int64_t)cu_seqlens[s + 1] - cu_seqlens[s];
        if (L < 0) return -1;
        n_items += H * ((L + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM);
    }
    if (n_items == 0) return 0;
    work_item *items = (work_item *)malloc(sizeof(work_item) * (size_t)n_items);
    if (!items) return -2;
    int64_t n = 0;
    for (int64_t s = 0; s < num_seqs; ++s) {
        int64_t start = cu_seqlens[s];
        int64_t L = (int64_t)cu_seqlens[s + 1] - start;
        int64_t chunks = (L + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM;
        for (int64_t h = 0; h < H; ++h)
            for (int64_t ch = 0; ch < chunks; ++ch) {
                work_item *w = &items[n++];
                w->q = q + (start * H + h) * d;
                w->k = k + (start * Hkv + h / G) * d;
                w->v = v + (start * Hkv + h / G) * d;
                w->row_stride = H * d;
                w->kv_row_stride = Hkv * d;
                w->nq = L; w->nkv = L; w->off = 0;
                w->o = o + (start * H + h) * d;
                w->lse = lse + h * T + start;
                w->row_begin = ch * ROWS_PER_ITEM;
                w->row_end = w->row_begin + ROWS_PER_ITEM < L ? w->row_begin + ROWS_PER_ITEM : L;
            }
    }
    int rc = run_pool(items, n_items, d, scale, causal, dtype, nthreads);
    free(items);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Selected rows only, for checks at sizes where the full oracle is too slow.
 * rows: n_rows triples (b, h, i) for the fixed-length layout.
 * o_rows [n_rows, d], lse_rows [n_rows].                                     */
typedef struct {
    const uint16_t *q, *k, *v;
    int64_t H, Hkv, Nq, Nkv, d, off;
    double scale;
    int causal;
    int dtype;
    const int64_t *rows;   /* triples (b,h,i), or (seq-start, h, local row, L) quads for varlen */
    int varlen;
    const int32_t *cu;
    int64_t n_rows;
    double *o_rows, *lse_rows;
    int64_t next;
    int failed;
} rows_job;

static void *rows_worker(void *arg)
{
    rows_job *J = (rows_job *)arg;
    int64_t d = J->d;
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);
    double *kd = NULL, *vd = NULL, *t = NULL;
    int64_t cap = 0;
    if (!qd) { __atomic_store_n(&J->failed, 1, __ATOMIC_RELAXED); return NULL; }
    for (;;) {
        int64_t r = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (r >= J->n_rows) break;
        const uint16_t *qb, *kb, *vb;
        int64_t i, nvalid, stride = J->H * d, kv_stride = J->Hkv * d, G = J->H / J->Hkv;
        if (!J->varlen) {
            int64_t b = J->rows[3 * r], h = J->rows[3 * r + 1];
            i = J->rows[3 * r + 2];
            qb = J->q + (b * J->Nq * J->H + h) * d;
            kb = J->k + (b * J->Nkv * J->Hkv + h / G) * d;
            vb = J->v + (b * J->Nkv * J->Hkv + h / G) * d;
            nvalid = valid_keys(i, J->Nkv, J->causal, J->off);
        } else {
            /* rows: pairs (h, token); find the token's sequence */
            int64_t h = J->rows[2 * r], tok = J->rows[2 * r + 1];
            int64_t lo = 0, hi = J->Nq; /* Nq holds num_seqs here */
            while (hi - lo > 1) {
                int64_t mid = (lo + hi) / 2;
                if (J->cu[mid] <= tok) lo = mid; else hi = mid;
            }
            int64_t start = J->cu[lo], L = (int64_t)J->cu[lo + 1] - start;
            i = tok - start;
            qb = J->q + (start * J->H + h) * d;
            kb = J->k + (start * J->Hkv + h / G) * d;
            vb = J->v + (start * J->Hkv + h / G) * d;
            nvalid = valid_keys(i, L, J->causal, 0);
        }
        if (nvalid > cap) {
            free(kd); free(vd); free(t);
            cap = nvalid;
            kd = (double *)malloc(sizeof(double) * (size_t)(cap * d));
            vd = (double *)malloc(sizeof(double) * (size_t)(cap * d));
            t = (double *)malloc(sizeof(double) * (size_t)cap);
            if (!kd || !vd || !t) { __atomic_store_n(&J->failed, 1, __ATOMIC_RELAXED); break; }
        }
        for (int64_t j = 0; j < nvalid; ++j)
            for (int64_t c = 0; c < d; ++c) {
                kd[j * d + c] = to_double(kb[j * kv_stride + c], J->dtype);
                vd[j * d + c] = to_double(vb[j * kv_stride + c], J->dtype);
            }
        for (int64_t c = 0; c < d; ++c) qd[c] = to_double(qb[i * stride + c], J->dtype);
        attend_row(qd, kd, vd, nvalid, d, J->scale, t ? t : qd, J->o_rows + r * d, J->lse_rows + r);
    }
    free(qd); free(kd); free(vd); free(t);
    return NULL;
}

static int run_rows(rows_job *J, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -2;
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, rows_worker, J) != 0) break;
        ++started;
    }
    rows_worker(J);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    free(th);
    return J->failed ? -2 : 0;
}

int oracle_attention_rows_bshd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               int64_t B, int64_t H, int64_t Hkv, int64_t Nq, int64_t Nkv,
                               int64_t d, int dtype, double scale, int causal, int64_t off,
                               const int64_t *rows, int64_t n_rows,
                               double *o_rows, double *lse_rows, int nthreads)
{
    if (!q || !k || !v || !rows || !o_rows || !lse_rows || d <= 0 || n_rows < 0 ||
        !heads_ok(H, Hkv, dtype))
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= Nq) return -1;
    }
    rows_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.H = H; J.Hkv = Hkv; J.Nq = Nq; J.Nkv = Nkv; J.d = d; J.off = off;
    J.scale = scale; J.causal = causal; J.dtype = dtype; J.rows = rows; J.varlen = 0;
    J.n_rows = n_rows; J.o_rows = o_rows; J.lse_rows = lse_rows;
    return run_rows(&J, nthreads);
}

/* rows: n_rows pairs (h, token) of the packed layout. */
int oracle_attention_rows_varlen(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const int32_t *cu_seqlens, int64_t num_seqs,
                                 int64_t H, int64_t Hkv, int64_t d, int dtype, double scale,
                                 int causal, const int64_t *rows, int64_t n_rows,
                                 double *o_rows, double *lse_rows, int nthreads)
{
    if (!q || !k || !v || !cu_seqlens || !rows || !o_rows || !lse_rows || d <= 0 ||
        num_seqs <= 0 || n_rows < 0 || !heads_ok(H, Hkv, dtype))
        return -1;
    int64_t T = cu_seqlens[num_seqs];
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t h = rows[2 * r], tok = rows[2 * r + 1];
        if (h < 0 || h >= H || tok < 0 || tok >= T) return -1;
    }
    rows_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.H = H; J.Hkv = Hkv; J.Nq = num_seqs; J.d = d;
    J.scale = scale; J.causal = causal; J.dtype = dtype; J.rows = rows; J.varlen = 1;
    J.cu = cu_seqlens;
    J.n_rows = n_rows; J.o_rows = o_rows; J.lse_rows = lse_rows;
    return run_rows(&J, nthreads);
}

/*
 * fp64 CPU oracle for fused scaled-dot-product attention with grouped KV heads.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library path uses this file: only the
 * tests, the package smoke check and the CPU-baseline leg of the benchmark load it.
 * It shares no code, header or table with the CUDA kernels.
 *
 * What it computes is the plain definition of masked softmax attention, one query
 * row at a time, with no blocking, no online rescaling and no score matrix:
 *
 *   s_ij  = scale * sum_d q[i,h,d] k[j,g,d]              g = h / (Hq / Hkv)
 *   allow(i,j) = (!causal || j <= i) && (window <= 0 || i - j < window)
 *   m_i   = max_{allowed j} s_ij,  l_i = sum_{allowed j} exp(s_ij - m_i)
 *   p_ij  = exp(s_ij - m_i) / l_i  (0 where not allowed)
 *   o_i   = sum_j p_ij v_j,   lse_i = m_i + ln l_i
 *
 * and its analytic gradient for an upstream gradient dO of o:
 *
 *   dp_ij = dO_i . v_j,   Delta_i = sum_j p_ij dp_ij,   ds_ij = p_ij (dp_ij - Delta_i)
 *   dq_i  = scale sum_j ds_ij k_j
 *   dk_j  = scale sum_{h in group} sum_i ds_ij q_i,   dv_j = sum_{h in group} sum_i p_ij dO_i
 *
 * Sources, by page and section:
 *  - "Gemma4 FFPA attention backend support ..." (NeMo-Automodel discussion 2928),
 *    operator table and "Debugging notes": the fused kernels compute the same
 *    attention as the MATH path that materialises the S x S score matrix; GQA is
 *    the repeat-KV mapping (each KV head serves a contiguous group of query heads);
 *    "Integration": a 2-D padding mask is served by the varlen path, i.e. each
 *    packed sequence is its own causal problem.
 *  - "flex_attention + paged KV + CUDA graphs vs vLLM", "What each option did" and
 *    "Architecture notes": a paged cache is the contiguous cache read through a
 *    page table; "What broke correctness": a row with no allowed key must not
 *    produce NaN (here: o = 0, lse = -inf).
 *  - Sliding window of width W: query i sees keys i-W+1 .. i (the window workload
 *    states keys i-1023..i for W = 1024).
 *
 * bf16 inputs are raw bit patterns, widened exactly to double.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one known mistake; it exists only
 * so a test can show that the pins catch each kind of mistake.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

static inline double bf16d(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ---------------------------------------------------------------------------------- */
/* One causal problem over a single sequence: rows of q/dO are [L, Hq, D], k/v [L, Hkv, D]. */
typedef struct {
    const uint16_t *q, *k, *v, *dO;
    int L, Hq, Hkv, D;
    double scale;
    int causal, window;
    int q_single; /* 1: q holds one row per head (a decode query), whatever i is */
    int q_first;  /* position of q's first row (the new queries of a paged prefill); 0 otherwise */
} seq_view;

static inline int kv_head_of(const seq_view* sv, int h) {
#if ORACLE_MUTANT == 2
    return h % sv->Hkv; /* planted: interleaved instead of contiguous head groups */
#else
    return h / (sv->Hq / sv->Hkv);
#endif
}

static inline int allowed(const seq_view* sv, int i, int j) {
    if (j < 0 || j >= sv->L) return 0;
#if ORACLE_MUTANT == 7
    if (sv->causal && j >= i) return 0; /* planted: diagonal excluded */
#else
    if (sv->causal && j > i) return 0;
#endif
#if ORACLE_MUTANT == 3
    if (sv->window > 0 && i - j > sv->window) return 0; /* planted: window one too wide */
#else
    if (sv->window > 0 && i - j >= sv->window) return 0;
#endif
    return 1;
}

static inline const uint16_t* qrow(const seq_view* sv, int i, int h) {
    if (sv->q_single) i = 0;
    else i -= sv->q_first;
    return sv->q + ((size_t)i * sv->Hq + h) * sv->D;
}
static inline const uint16_t* dorow(const seq_view* sv, int i, int h) { return sv->dO + ((size_t)i * sv->Hq + h) * sv->D; }
static inline const uint16_t* krow(const seq_view* sv, int j, int g) { return sv->k + ((size_t)j * sv->Hkv + g) * sv->D; }
static inline const uint16_t* vrow(const seq_view* sv, int j, int g) { return sv->v + ((size_t)j * sv->Hkv + g) * sv->D; }

static double dot_bf16(const uint16_t* a, const uint16_t* b, int D) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += bf16d(a[d]) * bf16d(b[d]);
    return acc;
}

/*
 * Softmax statistics of query row i of head h: fills s[j] for all j (0 where not
 * allowed), returns the number of allowed keys, sets *m and *l.
 */
static int row_scores(const seq_view* sv, int h, int i, double* s, double* m, double* l) {
    int g = kv_head_of(sv, h);
    int n = 0;
    double mx = -INFINITY;
    for (int j = 0; j < sv->L; ++j) {
        if (!allowed(sv, i, j)) {
            s[j] = 0.0;
            continue;
        }
        s[j] = sv->scale * dot_bf16(qrow(sv, i, h), krow(sv, j, g), sv->D);
        if (s[j] > mx) mx = s[j];
        ++n;
    }
    double sum = 0.0;
    if (n > 0)
        for (int j = 0; j < sv->L; ++j)
            if (allowed(sv, i, j)) sum += exp(s[j] - mx);
    *m = mx;
    *l = sum;
    return n;
}

/* Forward of one row: o (D doubles) and lse. s is scratch of L doubles. */
static void row_forward(const seq_view* sv, int h, int i, double* s, double* o, double* lse) {
    double m, l;
    int n = row_scores(sv, h, i, s, &m, &l);
    for (int d = 0; d < sv->D; ++d) o[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    int g = kv_head_of(sv, h);
    for (int j = 0; j < sv->L; ++j) {
        if (!allowed(sv, i, j)) continue;
        double p = exp(s[j] - m) / l;
        const uint16_t* vj = vrow(sv, j, g);
        for (int d = 0; d < sv->D; ++d) o[d] += p * bf16d(vj[d]);
    }
#if ORACLE_MUTANT == 5
    *lse = log(l); /* planted: max term dropped */
#else
    *lse = m + log(l);
#endif
}

/*
 * Backward pieces of one row: p[j], dp[j] for allowed j, Delta. Returns number of
 * allowed keys. Also returns Delta computed the second way (dO . o) in *delta_alt.
 */
static int row_backward_terms(const seq_view* sv, int h, int i, double* s, double* p, double* dp, double* o,
                              double* delta, double* delta_alt, double* m_out, double* l_out) {
    double m, l;
    int n = row_scores(sv, h, i, s, &m, &l);
    if (m_out) *m_out = m;
    if (l_out) *l_out = l;
    int g = kv_head_of(sv, h);
    double dl = 0.0;
    for (int d = 0; d < sv->D; ++d) o[d] = 0.0;
    for (int j = 0; j < sv->L; ++j) {
        if (!allowed(sv, i, j)) {
            p[j] = 0.0;
            dp[j] = 0.0;
            continue;
        }
        p[j] = exp(s[j] - m) / l;
        dp[j] = dot_bf16(dorow(sv, i, h), vrow(sv, j, g), sv->D);
        dl += p[j] * dp[j];
        const uint16_t* vj = vrow(sv, j, g);
        for (int d = 0; d < sv->D; ++d) o[d] += p[j] * bf16d(vj[d]);
    }
    double alt = 0.0;
    const uint16_t* doi = dorow(sv, i, h);
    for (int d = 0; d < sv->D; ++d) alt += bf16d(doi[d]) * o[d];
    *delta = dl;
    *delta_alt = alt;
    return n;
}

static inline double ds_of(double p, double dp, double delta) {
#if ORACLE_MUTANT == 1
    (void)delta;
    return p * dp; /* planted: softmax Jacobian's Delta term dropped */
#else
    return p * (dp - delta);
#endif
}

/* ---------------------------------------------------------------------------------- */
/* Minimal parallel-for over work items. */
typedef struct {
    atomic_long next;
    long count;
    void (*fn)(void* ctx, long item, double* scratch);
    void* ctx;
    size_t scratch_doubles;
    atomic_int failed;
} pfor_t;

static void* pfor_worker(void* arg) {
    pfor_t* pf = (pfor_t*)arg;
    double* scratch = (double*)malloc(sizeof(double) * (pf->scratch_doubles ? pf->scratch_doubles : 1));
    if (!scratch) {
        atomic_store(&pf->failed, 1);
        return NULL;
    }
    for (;;) {
        long it = atomic_fetch_add(&pf->next, 1);
        if (it >= pf->count) break;
        pf->fn(pf->ctx, it, scratch);
    }
    free(scratch);
    return NULL;
}

static int parallel_for(long count, int nthreads, size_t scratch_doubles, void (*fn)(void*, long, double*), void* ctx) {
    pfor_t pf;
    atomic_init(&pf.next, 0);
    atomic_init(&pf.failed, 0);
    pf.count = count;
    pf.fn = fn;
    pf.ctx = ctx;
    pf.scratch_doubles = scratch_doubles;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nthreads > count) nthreads = count > 0 ? (int)count : 1;
    pthread_t th[512];
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[started], NULL, pfor_worker, &pf) == 0) ++started;
    }
    pfor_worker(&pf);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    return atomic_load(&pf.failed) ? -2 : 0;
}

/* ---------------------------------------------------------------------------------- */
/* Dense [B, S, H, D] problems and packed varlen [T, H, D] problems share one driver:
 * a list of sequences, each with its token offset and length. */
typedef struct {
    const uint16_t *q, *k, *v, *dO;
    int Hq, Hkv, D;
    double scale;
    int causal, window;
    int nseq;
    const int64_t* off; /* token offset of sequence s */
    const int64_t* len; /* length of sequence s */
    int64_t T;          /* total tokens (lse stride) */
    /* outputs */
    double *o, *lse, *dq, *dk, *dv, *delta;
    double* gap; /* per work item max |Delta - dO.o| */
    int lse_layout_dense; /* 1: lse [B, Hq, S] with S = len (equal lengths); 0: [Hq, T] */
} problem_t;

static seq_view view_of(const problem_t* P, int s) {
    seq_view sv;
    size_t off = (size_t)P->off[s];
    sv.q = P->q + off * P->Hq * P->D;
    sv.k = P->k + off * P->Hkv * P->D;
    sv.v = P->v + off * P->Hkv * P->D;
    sv.dO = P->dO ? P->dO + off * P->Hq * P->D : NULL;
    sv.L = (int)P->len[s];
    sv.Hq = P->Hq;
    sv.Hkv = P->Hkv;
    sv.D = P->D;
    sv.scale = P->scale;
    sv.causal = P->causal;
    sv.window = P->window;
    sv.q_single = 0;
    sv.q_first = 0;
    return sv;
}

static size_t lse_index(const problem_t* P, int s, int h, int i) {
    if (P->lse_layout_dense) return ((size_t)s * P->Hq + h) * (size_t)P->len[s] + i;
    return (size_t)h * (size_t)P->T + (size_t)P->off[s] + i;
}

static void fwd_item(void* ctx, long item, double* scratch) {
    const problem_t* P = (const problem_t*)ctx;
    int s = (int)(item / P->Hq), h = (int)(item % P->Hq);
    seq_view sv = view_of(P, s);
    for (int i = 0; i < sv.L; ++i) {
        double* o = P->o + (((size_t)P->off[s] + i) * P->Hq + h) * P->D;
        double lse;
        row_forward(&sv, h, i, scratch, o, &lse);
        P->lse[lse_index(P, s, h, i)] = lse;
    }
}

static void bwd_item(void* ctx, long item, double* scratch) {
    const problem_t* P = (const problem_t*)ctx;
    int s = (int)(item / P->Hkv), g = (int)(item % P->Hkv);
    seq_view sv = view_of(P, s);
    int G = P->Hq / P->Hkv, D = P->D, L = sv.L;
    double* sb = scratch;
    double* p = sb + L;
    double* dp = p + L;
    double* o = dp + L;
    double gap = 0.0;
    size_t off = (size_t)P->off[s];
    for (int j = 0; j < L; ++j)
        for (int d = 0; d < D; ++d) {
            P->dk[((off + j) * P->Hkv + g) * D + d] = 0.0;
            P->dv[((off + j) * P->Hkv + g) * D + d] = 0.0;
        }
    for (int hh = 0; hh < G; ++hh) {
        int h = g * G + hh;
#if ORACLE_MUTANT == 2
        /* with the planted head mapping, the heads served by g are those with h % Hkv == g */
        h = hh * P->Hkv + g;
#endif
        for (int i = 0; i < L; ++i) {
            double delta, alt;
            int n = row_backward_terms(&sv, h, i, sb, p, dp, o, &delta, &alt, NULL, NULL);
            double* dqi = P->dq + ((off + i) * P->Hq + h) * D;
            for (int d = 0; d < D; ++d) dqi[d] = 0.0;
            if (P->o) {
                double* oo = P->o + ((off + i) * P->Hq + h) * D;
                for (int d = 0; d < D; ++d) oo[d] = o[d];
            }
            if (P->delta) P->delta[lse_index(P, s, h, i)] = delta;
            if (n == 0) continue;
            double gg = fabs(delta - alt);
            if (gg > gap) gap = gg;
            const uint16_t* qi = qrow(&sv, i, h);
            const uint16_t* doi = dorow(&sv, i, h);
            for (int j = 0; j < L; ++j) {
                if (!allowed(&sv, i, j)) continue;
                double ds = ds_of(p[j], dp[j], delta);
                const uint16_t* kj = krow(&sv, j, g);
                double* dkj = P->dk + ((off + j) * P->Hkv + g) * D;
                double* dvj = P->dv + ((off + j) * P->Hkv + g) * D;
                for (int d = 0; d < D; ++d) {
#if ORACLE_MUTANT == 8
                    dqi[d] += P->scale * ds * bf16d(vrow(&sv, j, g)[d]); /* planted: wrong operand */
#else
                    dqi[d] += P->scale * ds * bf16d(kj[d]);
#endif
#if ORACLE_MUTANT == 4
                    dkj[d] += ds * bf16d(qi[d]); /* planted: scale dropped */
#else
                    dkj[d] += P->scale * ds * bf16d(qi[d]);
#endif
#if ORACLE_MUTANT == 6
                    dvj[d] += ds * bf16d(doi[d]); /* planted: ds in place of p */
#else
                    dvj[d] += p[j] * bf16d(doi[d]);
#endif
                }
            }
        }
    }
    P->gap[item] = gap;
}

static int check_heads(int Hq, int Hkv, int D) {
    if (Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return -1;
    return 0;
}

static int run_fwd(problem_t* P, int nthreads) {
    int64_t maxL = 1;
    for (int s = 0; s < P->nseq; ++s)
        if (P->len[s] > maxL) maxL = P->len[s];
    return parallel_for((long)P->nseq * P->Hq, nthreads, (size_t)maxL, fwd_item, P);
}

static int run_bwd(problem_t* P, int nthreads, double* max_gap) {
    int64_t maxL = 1;
    for (int s = 0; s < P->nseq; ++s)
        if (P->len[s] > maxL) maxL = P->len[s];
    long items = (long)P->nseq * P->Hkv;
    P->gap = (double*)calloc((size_t)items, sizeof(double));
    if (!P->gap) return -2;
    int rc = parallel_for(items, nthreads, (size_t)(3 * maxL + P->D), bwd_item, P);
    double g = 0.0;
    for (long it = 0; it < items; ++it)
        if (P->gap[it] > g) g = P->gap[it];
    if (max_gap) *max_gap = g;
    free(P->gap);
    return rc;
}

/* ---------------------------------------------------------------------------------- */
/* Public entry points (ctypes). Outputs are doubles in the same layouts as the inputs;
 * lse is [B, Hq, S] (dense) or [Hq, T] (varlen). Return 0, or -1 on bad arguments. */

static int dense_problem(problem_t* P, int64_t** offs, int B, int S) {
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)(B > 0 ? B : 1));
    if (!off) return -2;
    for (int b = 0; b < B; ++b) {
        off[b] = (int64_t)b * S;
        off[B + b] = S;
    }
    P->nseq = B;
    P->off = off;
    P->len = off + B;
    P->T = (int64_t)B * S;
    P->lse_layout_dense = 1;
    *offs = off;
    return 0;
}

int oracle_attn_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int Hq, int Hkv, int S, int D,
                    double scale, int causal, int window, double* o, double* lse, int nthreads) {
    if (check_heads(Hq, Hkv, D) || B < 0 || S < 0) return -1;
    problem_t P = {0};
    P.q = q, P.k = k, P.v = v, P.Hq = Hq, P.Hkv = Hkv, P.D = D, P.scale = scale, P.causal = causal, P.window = window;
    P.o = o, P.lse = lse;
    int64_t* offs;
    if (dense_problem(&P, &offs, B, S)) return -2;
    int rc = run_fwd(&P, nthreads);
    free(offs);
    return rc;
}

int oracle_attn_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dO, int B, int Hq, int Hkv,
                    int S, int D, double scale, int causal, int window, double* dq, double* dk, double* dv, double* o,
                    double* delta, double* max_delta_gap, int nthreads) {
    if (check_heads(Hq, Hkv, D) || B < 0 || S < 0 || !dO) return -1;
    problem_t P = {0};
    P.q = q, P.k = k, P.v = v, P.dO = dO, P.Hq = Hq, P.Hkv = Hkv, P.D = D, P.scale = scale, P.causal = causal;
    P.window = window, P.dq = dq, P.dk = dk, P.dv = dv, P.o = o, P.delta = delta;
    int64_t* offs;
    if (dense_problem(&P, &offs, B, S)) return -2;
    int rc = run_bwd(&P, nthreads, max_delta_gap);
    free(offs);
    return rc;
}

static int varlen_problem(problem_t* P, int64_t** offs, const int32_t* cu, int nseq) {
    if (nseq < 0 || !cu || cu[0] != 0) return -1;
    for (int s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s]) return -1;
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)(nseq > 0 ? nseq : 1));
    if (!off) return -2;
    for (int s = 0; s < nseq; ++s) {
        off[s] = cu[s];
        off[nseq + s] = (int64_t)cu[s + 1] - cu[s];
    }
    P->nseq = nseq;
    P->off = off;
    P->len = off + nseq;
    P->T = cu[nseq];
    P->lse_layout_dense = 0;
    *offs = off;
    return 0;
}

int oracle_attn_fwd_varlen(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* cu_seqlens, int num_seqs,
                           int Hq, int Hkv, int D, double scale, int causal, int window, double* o, double* lse,
                           int nthreads) {
    if (check_heads(Hq, Hkv, D)) return -1;
    problem_t P = {0};
    P.q = q, P.k = k, P.v = v, P.Hq = Hq, P.Hkv = Hkv, P.D = D, P.scale = scale, P.causal = causal, P.window = window;
    P.o = o, P.lse = lse;
    int64_t* offs;
    int rc = varlen_problem(&P, &offs, cu_seqlens, num_seqs);
    if (rc) return rc;
    rc = run_fwd(&P, nthreads);
    free(offs);
    return rc;
}

int oracle_attn_bwd_varlen(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dO,
                           const int32_t* cu_seqlens, int num_seqs, int Hq, int Hkv, int D, double scale, int causal,
                           int window, double* dq, double* dk, double* dv, double* max_delta_gap, int nthreads) {
    if (check_heads(Hq, Hkv, D) || !dO) return -1;
    problem_t P = {0};
    P.q = q, P.k = k, P.v = v, P.dO = dO, P.Hq = Hq, P.Hkv = Hkv, P.D = D, P.scale = scale, P.causal = causal;
    P.window = window, P.dq = dq, P.dk = dk, P.dv = dv;
    int64_t* offs;
    int rc = varlen_problem(&P, &offs, cu_seqlens, num_seqs);
    if (rc) return rc;
    rc = run_bwd(&P, nthreads, max_delta_gap);
    free(offs);
    return rc;
}

/* ---------------------------------------------------------------------------------- */
/* Sampled rows of a dense problem, for workloads too large to compute whole. */
typedef struct {
    problem_t P;
    const int64_t* rows; /* triples */
    double *out_a, *out_b;
} rows_ctx;

static void fwd_rows_item(void* ctx, long r, double* scratch) {
    rows_ctx* C = (rows_ctx*)ctx;
    int b = (int)C->rows[3 * r], h = (int)C->rows[3 * r + 1], i = (int)C->rows[3 * r + 2];
    seq_view sv = view_of(&C->P, b);
    row_forward(&sv, h, i, scratch, C->out_a + (size_t)r * C->P.D, C->out_b + r);
}

static void dq_rows_item(void* ctx, long r, double* scratch) {
    rows_ctx* C = (rows_ctx*)ctx;
    int b = (int)C->rows[3 * r], h = (int)C->rows[3 * r + 1], i = (int)C->rows[3 * r + 2];
    seq_view sv = view_of(&C->P, b);
    int L = sv.L, D = sv.D, g = kv_head_of(&sv, h);
    double *s = scratch, *p = s + L, *dp = p + L, *o = dp + L;
    double delta, alt;
    double* dq = C->out_a + (size_t)r * D;
    for (int d = 0; d < D; ++d) dq[d] = 0.0;
    if (row_backward_terms(&sv, h, i, s, p, dp, o, &delta, &alt, NULL, NULL) == 0) return;
    for (int j = 0; j < L; ++j) {
        if (!allowed(&sv, i, j)) continue;
        double ds = ds_of(p[j], dp[j], delta);
        const uint16_t* kj = krow(&sv, j, g);
        for (int d = 0; d < D; ++d) dq[d] += sv.scale * ds * bf16d(kj[d]);
    }
}

/* rows: (sequence b, query head h, query i) triples into a dense [B,S,..] or varlen problem. */
static int rows_common(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dO,
                       const int32_t* cu_seqlens, int nseq_or_B, int S, int Hq, int Hkv, int D, double scale, int causal,
                       int window, rows_ctx* C, int64_t** offs) {
    if (check_heads(Hq, Hkv, D)) return -1;
    memset(&C->P, 0, sizeof(C->P));
    C->P.q = q, C->P.k = k, C->P.v = v, C->P.dO = dO, C->P.Hq = Hq, C->P.Hkv = Hkv, C->P.D = D;
    C->P.scale = scale, C->P.causal = causal, C->P.window = window;
    if (cu_seqlens) return varlen_problem(&C->P, offs, cu_seqlens, nseq_or_B);
    return dense_problem(&C->P, offs, nseq_or_B, S);
}

static int rows_check(const rows_ctx* C, const int64_t* rows, long nrows, int head_limit) {
    for (long r = 0; r < nrows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= C->P.nseq || h < 0 || h >= head_limit || i < 0 || i >= C->P.len[b]) return -1;
    }
    return 0;
}

int oracle_attn_fwd_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* cu_seqlens, int nseq_or_B,
                         int S, int Hq, int Hkv, int D, double scale, int causal, int window, const int64_t* rows,
                         long nrows, double* o, double* lse, int nthreads) {
    rows_ctx C;
    int64_t* offs;
    int rc = rows_common(q, k, v, NULL, cu_seqlens, nseq_or_B, S, Hq, Hkv, D, scale, causal, window, &C, &offs);
    if (rc) return rc;
    if (rows_check(&C, rows, nrows, Hq)) {
        free(offs);
        return -1;
    }
    C.rows = rows, C.out_a = o, C.out_b = lse;
    int64_t maxL = 1;
    for (int s = 0; s < C.P.nseq; ++s)
        if (C.P.len[s] > maxL) maxL = C.P.len[s];
    rc = parallel_for(nrows, nthreads, (size_t)maxL, fwd_rows_item, &C);
    free(offs);
    return rc;
}

int oracle_attn_dq_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dO,
                        const int32_t* cu_seqlens, int nseq_or_B, int S, int Hq, int Hkv, int D, double scale, int causal,
                        int window, const int64_t* rows, long nrows, double* dq, int nthreads) {
    rows_ctx C;
    int64_t* offs;
    if (!dO) return -1;
    int rc = rows_common(q, k, v, dO, cu_seqlens, nseq_or_B, S, Hq, Hkv, D, scale, causal, window, &C, &offs);
    if (rc) return rc;
    if (rows_check(&C, rows, nrows, Hq)) {
        free(offs);
        return -1;
    }
    C.rows = rows, C.out_a = dq;
    int64_t maxL = 1;
    for (int s = 0; s < C.P.nseq; ++s)
        if (C.P.len[s] > maxL) maxL = C.P.len[s];
    rc = parallel_for(nrows, nthreads, (size_t)(3 * maxL + D), dq_rows_item, &C);
    free(offs);
    return rc;
}

/*
 * dK and dV rows (b, kv head g, key j). Every query row that sees key j contributes,
 * so the softmax statistics (m, l, Delta) of those rows are computed first, once per
 * (b, h, i) that any requested key needs, then each requested key row is summed.
 */
typedef struct {
    rows_ctx* C;
    /* per needed query row: */
    long nq;
    const int64_t* qrows; /* (b, h, i) */
    double *m, *l, *delta;
} dkv_stats_ctx;

static void dkv_stats_item(void* ctx, long r, double* scratch) {
    dkv_stats_ctx* X = (dkv_stats_ctx*)ctx;
    int b = (int)X->qrows[3 * r], h = (int)X->qrows[3 * r + 1], i = (int)X->qrows[3 * r + 2];
    seq_view sv = view_of(&X->C->P, b);
    int L = sv.L;
    double *s = scratch, *p = s + L, *dp = p + L, *o = dp + L;
    double delta, alt, m, l;
    row_backward_terms(&sv, h, i, s, p, dp, o, &delta, &alt, &m, &l);
    X->m[r] = m;
    X->l[r] = l;
    X->delta[r] = delta;
}

typedef struct {
    rows_ctx* C;
    dkv_stats_ctx* X;
    const int64_t* first; /* per (b, h): index into qrows of query 0 of that (b,h), or -1 */
    int Hq;
} dkv_acc_ctx;

static void dkv_acc_item(void* ctx, long r, double* scratch) {
    (void)scratch;
    dkv_acc_ctx* A = (dkv_acc_ctx*)ctx;
    rows_ctx* C = A->C;
    int b = (int)C->rows[3 * r], g = (int)C->rows[3 * r + 1], j = (int)C->rows[3 * r + 2];
    seq_view sv = view_of(&C->P, b);
    int D = sv.D, G = sv.Hq / sv.Hkv;
    double* dk = C->out_a + (size_t)r * D;
    double* dv = C->out_b + (size_t)r * D;
    for (int d = 0; d < D; ++d) dk[d] = dv[d] = 0.0;
    const uint16_t* kj = krow(&sv, j, g);
    const uint16_t* vj = vrow(&sv, j, g);
    for (int h = 0; h < sv.Hq; ++h) {
        if (kv_head_of(&sv, h) != g) continue;
        (void)G;
        int64_t base = A->first[(size_t)b * A->Hq + h];
        for (int i = 0; i < sv.L; ++i) {
            if (!allowed(&sv, i, j)) continue;
            long qr = (long)(base + i);
            double s = sv.scale * dot_bf16(qrow(&sv, i, h), kj, D);
            double p = exp(s - A->X->m[qr]) / A->X->l[qr];
            double dp = dot_bf16(dorow(&sv, i, h), vj, D);
            double ds = ds_of(p, dp, A->X->delta[qr]);
            const uint16_t* qi = qrow(&sv, i, h);
            const uint16_t* doi = dorow(&sv, i, h);
            for (int d = 0; d < D; ++d) {
                dk[d] += sv.scale * ds * bf16d(qi[d]);
                dv[d] += p * bf16d(doi[d]);
            }
        }
    }
}

int oracle_attn_dkv_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dO,
                         const int32_t* cu_seqlens, int nseq_or_B, int S, int Hq, int Hkv, int D, double scale,
                         int causal, int window, const int64_t* rows, long nrows, double* dk, double* dv, int nthreads) {
    rows_ctx C;
    int64_t* offs;
    if (!dO) return -1;
    int rc = rows_common(q, k, v, dO, cu_seqlens, nseq_or_B, S, Hq, Hkv, D, scale, causal, window, &C, &offs);
    if (rc) return rc;
    if (rows_check(&C, rows, nrows, Hkv)) {
        free(offs);
        return -1;
    }
    C.rows = rows, C.out_a = dk, C.out_b = dv;
    int nseq = C.P.nseq;
    /* Query rows that can see a requested key: for every (b, h) whose KV head is
     * requested, the hull [min j, last row that sees max j] of the requested keys. */
    size_t nbh = (size_t)nseq * Hq;
    int64_t* first = (int64_t*)malloc(sizeof(int64_t) * nbh);
    int64_t* ilo = (int64_t*)malloc(sizeof(int64_t) * nbh);
    int64_t* ihi = (int64_t*)malloc(sizeof(int64_t) * nbh);
    char* need = (char*)calloc(nbh, 1);
    if (!first || !need || !ilo || !ihi) {
        free(first), free(need), free(ilo), free(ihi), free(offs);
        return -2;
    }
    seq_view sv0 = view_of(&C.P, 0);
    for (long r = 0; r < nrows; ++r) {
        int b = (int)rows[3 * r], g = (int)rows[3 * r + 1];
        int64_t j = rows[3 * r + 2], L = C.P.len[b];
        int64_t lo = C.P.causal ? j : 0;
        int64_t hi = (window > 0) ? j + window - 1 : L - 1;
        if (hi > L - 1) hi = L - 1;
        if (!C.P.causal) lo = (window > 0 && j - window + 1 > 0) ? j - window + 1 : 0;
        for (int h = 0; h < Hq; ++h) {
            if (kv_head_of(&sv0, h) != g) continue;
            size_t bh = (size_t)b * Hq + h;
            if (!need[bh]) {
                need[bh] = 1;
                ilo[bh] = lo;
                ihi[bh] = hi;
            } else {
                if (lo < ilo[bh]) ilo[bh] = lo;
                if (hi > ihi[bh]) ihi[bh] = hi;
            }
        }
    }
    long nq = 0;
    for (size_t bh = 0; bh < nbh; ++bh) {
        first[bh] = need[bh] ? nq - ilo[bh] : -1; /* index of row i is first[bh] + i */
        if (need[bh] && ihi[bh] >= ilo[bh]) nq += (long)(ihi[bh] - ilo[bh] + 1);
    }
    int64_t* qrows = (int64_t*)malloc(sizeof(int64_t) * 3 * (size_t)(nq > 0 ? nq : 1));
    double* st = (double*)malloc(sizeof(double) * 3 * (size_t)(nq > 0 ? nq : 1));
    if (!qrows || !st) {
        free(first), free(need), free(ilo), free(ihi), free(offs), free(qrows), free(st);
        return -2;
    }
    for (size_t bh = 0; bh < nbh; ++bh) {
        if (!need[bh]) continue;
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        for (int64_t i = ilo[bh]; i <= ihi[bh]; ++i) {
            long r = (long)(first[bh] + i);
            qrows[3 * r] = b, qrows[3 * r + 1] = h, qrows[3 * r + 2] = i;
        }
    }
    dkv_stats_ctx X = {&C, nq, qrows, st, st + nq, st + 2 * nq};
    int64_t maxL = 1;
    for (int s = 0; s < nseq; ++s)
        if (C.P.len[s] > maxL) maxL = C.P.len[s];
    rc = parallel_for(nq, nthreads, (size_t)(3 * maxL + D), dkv_stats_item, &X);
    if (rc == 0) {
        dkv_acc_ctx A = {&C, &X, first, Hq};
        rc = parallel_for(nrows, nthreads, 1, dkv_acc_item, &A);
    }
    free(first), free(need), free(ilo), free(ihi), free(offs), free(qrows), free(st);
    return rc;
}

/* ---------------------------------------------------------------------------------- */
/*
 * Single-token decode over a paged cache. Request b has L_b = seq_lens[b] cached
 * tokens; token t lives in page block_table[b][t / page_size], slot t % page_size, of
 * k_cache / v_cache [num_pages, page_size, Hkv, D]. The query sits at position
 * L_b - 1 and sees every cached token (bottom-right causal alignment), or the last
 * `window` of them when window > 0. Implemented literally: gather the request's
 * keys and values into a contiguous [L_b, Hkv, D] copy, then run the row forward.
 * Returns -1 on a page id outside the pool.
 */
typedef struct {
    const uint16_t *q, *kc, *vc;
    const int32_t *bt, *lens;
    int B, Hq, Hkv, D, ps, max_pages, num_pages, window;
    double scale;
    double *o, *lse;
    atomic_int bad;
} decode_ctx;

static void decode_item(void* ctx, long b, double* scratch) {
    decode_ctx* X = (decode_ctx*)ctx;
    int L = X->lens[b], D = X->D, Hkv = X->Hkv;
    size_t row = (size_t)Hkv * D;
    uint16_t* kk = (uint16_t*)malloc(sizeof(uint16_t) * row * (size_t)(L > 0 ? L : 1));
    uint16_t* vv = (uint16_t*)malloc(sizeof(uint16_t) * row * (size_t)(L > 0 ? L : 1));
    if (!kk || !vv) {
        free(kk), free(vv);
        atomic_store(&X->bad, 2);
        return;
    }
    for (int t = 0; t < L; ++t) {
        int pidx = t / X->ps;
        if (pidx >= X->max_pages) {
            atomic_store(&X->bad, 1);
            free(kk), free(vv);
            return;
        }
        int page = X->bt[(size_t)b * X->max_pages + pidx];
        if (page < 0 || page >= X->num_pages) {
            atomic_store(&X->bad, 1);
            free(kk), free(vv);
            return;
        }
        size_t src = ((size_t)page * X->ps + (size_t)(t % X->ps)) * row;
        memcpy(kk + (size_t)t * row, X->kc + src, sizeof(uint16_t) * row);
        memcpy(vv + (size_t)t * row, X->vc + src, sizeof(uint16_t) * row);
    }
    seq_view sv;
    sv.q = X->q + (size_t)b * X->Hq * D; /* the request's single query row [Hq, D] */
    sv.q_single = 1;
    sv.q_first = 0;
    sv.k = kk, sv.v = vv, sv.dO = NULL, sv.L = L, sv.Hq = X->Hq, sv.Hkv = Hkv, sv.D = D;
    sv.scale = X->scale, sv.causal = 1, sv.window = X->window;
    for (int h = 0; h < X->Hq; ++h) {
        double* o = X->o + ((size_t)b * X->Hq + h) * D;
        if (L == 0) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            X->lse[(size_t)b * X->Hq + h] = -INFINITY;
            continue;
        }
        row_forward(&sv, h, L - 1, scratch, o, &X->lse[(size_t)b * X->Hq + h]);
    }
    free(kk), free(vv);
}

int oracle_attn_decode_paged(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* block_table,
                             const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                             int num_pages, double scale, int window, double* o, double* lse, int nthreads) {
    if (check_heads(Hq, Hkv, D) || B < 0 || page_size <= 0 || max_pages < 0 || num_pages < 0) return -1;
    int maxL = 1;
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0) return -1;
        if (seq_lens[b] > maxL) maxL = seq_lens[b];
    }
    decode_ctx X = {q, k_cache, v_cache, block_table, seq_lens, B, Hq, Hkv, D, page_size, max_pages, num_pages, window,
                    scale, o, lse, 0};
    atomic_init(&X.bad, 0);
    int rc = parallel_for(B, nthreads, (size_t)maxL, decode_item, &X);
    if (rc) return rc;
    return atomic_load(&X.bad) ? -1 : 0;
}

/* ---------------------------------------------------------------------------------- */
/*
 * Prefill over a paged cache (chunked prefill): request b has L_b = seq_lens[b] cached
 * tokens (pages as in the decode above) and n_b = cu_q[b+1] - cu_q[b] new query tokens,
 * rows cu_q[b] .. cu_q[b+1]-1 of q [T, Hq, D], which are the last n_b of its L_b tokens
 * (their keys and values are already in the cache). New query i sits at position
 * L_b - n_b + i and sees the cached tokens at positions <= its own (and within the window).
 * The single-token decode is the case n_b = 1. Implemented literally: gather the request's
 * keys and values into a contiguous copy, then run the row forward for each new query.
 * Outputs o [T, Hq, D] and lse [Hq, T]. Returns -1 on a page id outside the pool or
 * n_b > L_b.
 */
typedef struct {
    const uint16_t *q, *kc, *vc;
    const int32_t *bt, *lens, *cu_q;
    int Hq, Hkv, D, ps, max_pages, num_pages, window;
    int64_t T;
    double scale;
    double *o, *lse;
    atomic_int bad;
} prefill_paged_ctx;

static void prefill_paged_item(void* ctx, long b, double* scratch) {
    prefill_paged_ctx* X = (prefill_paged_ctx*)ctx;
    const int L = X->lens[b], D = X->D, Hkv = X->Hkv;
    const int q0 = X->cu_q[b], nq = X->cu_q[b + 1] - X->cu_q[b];
    if (nq < 0 || nq > L) {
        atomic_store(&X->bad, 1);
        return;
    }
    if (nq == 0) return;
    size_t row = (size_t)Hkv * D;
    uint16_t* kk = (uint16_t*)malloc(sizeof(uint16_t) * row * (size_t)L);
    uint16_t* vv = (uint16_t*)malloc(sizeof(uint16_t) * row * (size_t)L);
    if (!kk || !vv) {
        free(kk), free(vv);
        atomic_store(&X->bad, 2);
        return;
    }
    for (int t = 0; t < L; ++t) {
        int pidx = t / X->ps;
        int page = pidx < X->max_pages ? X->bt[(size_t)b * X->max_pages + pidx] : -1;
        if (page < 0 || page >= X->num_pages) {
            atomic_store(&X->bad, 1);
            free(kk), free(vv);
            return;
        }
        size_t src = ((size_t)page * X->ps + (size_t)(t % X->ps)) * row;
        memcpy(kk + (size_t)t * row, X->kc + src, sizeof(uint16_t) * row);
        memcpy(vv + (size_t)t * row, X->vc + src, sizeof(uint16_t) * row);
    }
    seq_view sv;
    sv.q = X->q + (size_t)q0 * X->Hq * D; /* the request's new rows [nq, Hq, D] */
    sv.q_single = 0;
    sv.q_first = L - nq;
    sv.k = kk, sv.v = vv, sv.dO = NULL, sv.L = L, sv.Hq = X->Hq, sv.Hkv = Hkv, sv.D = D;
    sv.scale = X->scale, sv.causal = 1, sv.window = X->window;
    for (int i = 0; i < nq; ++i)
        for (int h = 0; h < X->Hq; ++h)
            row_forward(&sv, h, L - nq + i, scratch, X->o + ((size_t)(q0 + i) * X->Hq + h) * D,
                        &X->lse[(size_t)h * X->T + q0 + i]);
    free(kk), free(vv);
}

int oracle_attn_prefill_paged(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                              const int32_t* block_table, const int32_t* seq_lens, const int32_t* cu_q, int B, int Hq,
                              int Hkv, int D, int page_size, int max_pages, int num_pages, double scale, int window,
                              double* o, double* lse, int nthreads) {
    if (check_heads(Hq, Hkv, D) || B < 0 || page_size <= 0 || max_pages < 0 || num_pages < 0) return -1;
    int maxL = 1;
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0) return -1;
        if (seq_lens[b] > maxL) maxL = seq_lens[b];
    }
    prefill_paged_ctx X = {q, k_cache, v_cache, block_table, seq_lens, cu_q, Hq, Hkv, D, page_size, max_pages,
                           num_pages, window, (int64_t)cu_q[B], scale, o, lse, 0};
    atomic_init(&X.bad, 0);
    int rc = parallel_for(B, nthreads, (size_t)maxL, prefill_paged_item, &X);
    if (rc) return rc;
    return atomic_load(&X.bad) ? -1 : 0;
}

/*
 * Merge of attention results over disjoint key sets (the combining step of context-parallel
 * ring attention). "Gemma4 FFPA attention backend support ...", "Integration": under
 * context parallelism every ring chunk of keys is attended separately by the fused kernel
 * (dense or varlen per chunk) and the chunks' results make up the attention over all keys.
 * The pages do not write the combination out; it is the softmax over the union of the key
 * sets. Part p holds o_p, normalised over its own keys, and lse_p = ln sum_{j in p} exp(s_j):
 *
 *   lse = ln sum_p exp(lse_p),    o = sum_p exp(lse_p - lse) o_p
 *
 * evaluated with the largest lse_p factored out of the sum (exact algebra, no overflow).
 * A part with lse_p = -inf had no allowed key and contributes nothing; a row where every
 * part has lse_p = -inf gets o = 0 and lse = -inf.
 * Inputs o_parts [P, B, S, H, D] and lse_parts [P, B, H, S] in fp64; outputs o [B, S, H, D]
 * and lse [B, H, S].
 */
int oracle_merge_lse(const double* o_parts, const double* lse_parts, int P, int B, int S, int H, int D, double* o,
                     double* lse) {
    if (P < 1 || B < 0 || S < 0 || H < 1 || D < 1) return -1;
    const size_t rows = (size_t)B * S * H;
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < S; ++s)
            for (int h = 0; h < H; ++h) {
                const size_t orow = (((size_t)b * S + s) * H + h) * D;
                const size_t li = ((size_t)b * H + h) * S + s;
                double m = -INFINITY;
                for (int p = 0; p < P; ++p) {
                    const double x = lse_parts[(size_t)p * B * H * S + li];
                    if (x > m) m = x;
                }
                double* out = o + orow;
                for (int d = 0; d < D; ++d) out[d] = 0.0;
                if (m == -INFINITY) {
                    lse[li] = -INFINITY;
                    continue;
                }
                double sum = 0.0;
                for (int p = 0; p < P; ++p) {
#if ORACLE_MUTANT == 10
                    sum += exp(lse_parts[(size_t)p * B * H * S + li]); /* planted: no max factored out */
#else
                    sum += exp(lse_parts[(size_t)p * B * H * S + li] - m);
#endif
                }
#if ORACLE_MUTANT == 10
                const double L = log(sum);
#else
                const double L = m + log(sum);
#endif
                lse[li] = L;
                for (int p = 0; p < P; ++p) {
                    const double lp = lse_parts[(size_t)p * B * H * S + li];
                    if (lp == -INFINITY) continue;
#if ORACLE_MUTANT == 9
                    const double w = exp(L - lp); /* planted: weight with the sign flipped */
#else
                    const double w = exp(lp - L);
#endif
                    const double* src = o_parts + (size_t)p * rows * D + orow;
                    for (int d = 0; d < D; ++d) out[d] += w * src[d];
                }
            }
    return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }

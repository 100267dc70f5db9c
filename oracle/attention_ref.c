/*
 * Exact-attention oracle: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no header, helper or constant with the CUDA
 * library.
 *
 * What it computes, and where the pages define it:
 *
 *   oracle_attention_head / oracle_attention
 *     O = softmax(scale * Q K^T [+ causal mask]) V and LSE = log sum exp of the
 *     masked, scaled scores. S and P are materialised in full for every
 *     requested query row, exactly as the "Naive Attention" stage describes
 *     ("Adaptive High-Performance Attention Kernels in CUDA", Architectural
 *     Progression, Stage 1: S = QK^T and P = Softmax(S) materialised). The
 *     scale multiplies QK^T before the max and the exponential, as in the
 *     backward-pass recomputation S_ij = Q_i K_j^T / sqrt(d) (same page,
 *     Advanced Production Features 2). The causal rule keeps key k for query q
 *     iff k <= q ("FlashAttention-2 MMA", Technical Details, Causal Masking):
 *     top-left alignment, indices relative to the start of the sequence.
 *     The online-softmax tiling of the method reaches this same result up to
 *     rounding order, so the oracle is the plain definition, not the tiling.
 *
 *   oracle_splitkv_partials
 *     Phase 1 of split-K FlashDecoding ("Adaptive High-Performance Attention
 *     Kernels in CUDA", Advanced Production Features 1): the Sk keys of one
 *     head are cut into S partitions of ceil(Sk/S) keys (the last may be short
 *     or empty) and each partition yields an unnormalised partial output O_s,
 *     its score maximum m_s and its exponential sum l_s.
 *
 *   oracle_splitkv_merge
 *     Phase 2 of the same feature: O = sum_s e^{m_s - m_g} / l_g * O_s. The
 *     page leaves m_g and l_g undefined; the reading taken is m_g = max_s m_s
 *     and l_g = sum_s e^{m_s - m_g} l_s with O_s unnormalised, the only reading
 *     under which the printed sum equals full attention. LSE = m_g + ln l_g.
 *
 *   oracle_attention_bwd_head / oracle_attention_bwd
 *     Gradients of the loss L = sum(O * dO) with respect to Q, K and V for
 *     O = softmax(scale * Q K^T [+ causal mask]) V ("Adaptive High-Performance
 *     Attention Kernels in CUDA", Advanced Production Features 2, Custom CUDA
 *     Backward Pass): S and P are recomputed (here from scratch, in full),
 *     D_i = sum_k dO_ik O_ik, dS_ij = P_ij (dP_ij - D_i). The page names dS
 *     and D_i only; the remaining steps are the chain rule of the same
 *     definition: dV = P^T dO, dP = dO V^T, dQ = scale * dS K,
 *     dK = scale * dS^T Q.
 *
 * All arrays are row-major doubles owned by the caller. Return value 0 on
 * success, -1 on a bad argument, -2 on an allocation failure.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* One head. q: [Sq][D], k and v: [Sk][D]. rows: the nrows query indices to
 * evaluate (NULL means every row 0..Sq-1, and then nrows must equal Sq).
 * o: [nrows][D], lse: [nrows]. */
int oracle_attention_head(const double *q, const double *k, const double *v,
                          int Sq, int Sk, int D, int causal, double scale,
                          const int *rows, int nrows, double *o, double *lse)
{
    if (Sq < 1 || Sk < 1 || D < 1 || nrows < 0) return -1;
    if (rows == NULL && nrows != Sq) return -1;
    if (nrows == 0) return 0;

    double *S = (double *)malloc((size_t)nrows * (size_t)Sk * sizeof(double));
    double *P = (double *)malloc((size_t)nrows * (size_t)Sk * sizeof(double));
    if (!S || !P) { free(S); free(P); return -2; }

    for (int r = 0; r < nrows; ++r) {
        const int i = rows ? rows[r] : r;
        if (i < 0 || i >= Sq) { free(S); free(P); return -1; }

        /* S_ij = scale * q_i . k_j */
        for (int j = 0; j < Sk; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q[(size_t)i * D + d] * k[(size_t)j * D + d];
            S[(size_t)r * Sk + j] = scale * dot;
        }
        /* causal mask: key j is hidden from query i when j > i */
        if (causal)
            for (int j = i + 1; j < Sk; ++j) S[(size_t)r * Sk + j] = -INFINITY;

        /* m_i = max_j S_ij */
        double m = -INFINITY;
        for (int j = 0; j < Sk; ++j)
            if (S[(size_t)r * Sk + j] > m) m = S[(size_t)r * Sk + j];

        /* P_ij = exp(S_ij - m_i), l_i = sum_j P_ij, P_ij /= l_i */
        double l = 0.0;
        for (int j = 0; j < Sk; ++j) {
            P[(size_t)r * Sk + j] = exp(S[(size_t)r * Sk + j] - m);
            l += P[(size_t)r * Sk + j];
        }
        for (int j = 0; j < Sk; ++j) P[(size_t)r * Sk + j] /= l;

        /* O_i = sum_j P_ij v_j */
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int j = 0; j < Sk; ++j) acc += P[(size_t)r * Sk + j] * v[(size_t)j * D + d];
            o[(size_t)r * D + d] = acc;
        }
        /* LSE_i = m_i + ln l_i */
        lse[r] = m + log(l);
    }
    free(S);
    free(P);
    return 0;
}

/* ---- many heads, one worker thread per slice of heads ------------------- */

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int Sq, Sk, D, causal;
    double scale;
    const int *rows;
    int nrows;
    int head_begin, head_end;
    int status;
} heads_job;

static void *run_heads(void *arg)
{
    heads_job *jb = (heads_job *)arg;
    jb->status = 0;
    for (int h = jb->head_begin; h < jb->head_end && jb->status == 0; ++h) {
        jb->status = oracle_attention_head(
            jb->q + (size_t)h * jb->Sq * jb->D, jb->k + (size_t)h * jb->Sk * jb->D,
            jb->v + (size_t)h * jb->Sk * jb->D, jb->Sq, jb->Sk, jb->D, jb->causal,
            jb->scale, jb->rows, jb->nrows, jb->o + (size_t)h * jb->nrows * jb->D,
            jb->lse + (size_t)h * jb->nrows);
    }
    return NULL;
}

/* q: [BH][Sq][D], k and v: [BH][Sk][D], o: [BH][nrows][D], lse: [BH][nrows].
 * The same row list is evaluated in every head. */
int oracle_attention(const double *q, const double *k, const double *v, double *o,
                     double *lse, int BH, int Sq, int Sk, int D, int causal,
                     double scale, const int *rows, int nrows, int nthreads)
{
    if (BH < 0) return -1;
    if (BH == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > BH) nthreads = BH;

    heads_job *jobs = (heads_job *)calloc((size_t)nthreads, sizeof(heads_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -2; }

    for (int t = 0; t < nthreads; ++t) {
        heads_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->o = o; jb->lse = lse;
        jb->Sq = Sq; jb->Sk = Sk; jb->D = D; jb->causal = causal; jb->scale = scale;
        jb->rows = rows; jb->nrows = nrows;
        jb->head_begin = (int)((long long)BH * t / nthreads);
        jb->head_end = (int)((long long)BH * (t + 1) / nthreads);
    }
    int status = 0;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, run_heads, &jobs[t]) != 0) { status = -2; break; }
        ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    for (int t = 0; t < started && status == 0; ++t) status = jobs[t].status;
    free(jobs);
    free(tids);
    return status;
}

/* ---- split-K decoding, phase 1 ------------------------------------------- */

/* One head, one query. q: [D], k and v: [Sk][D]. Outputs per partition s:
 * o_part [S][D] (unnormalised), m_part [S], l_part [S]; an empty partition
 * gets m = -inf, l = 0, O = 0. Scores are in natural-log units of the scaled
 * dot product. */
int oracle_splitkv_partials(const double *q, const double *k, const double *v, int Sk,
                            int D, double scale, int num_splits, double *o_part,
                            double *m_part, double *l_part)
{
    if (Sk < 1 || D < 1 || num_splits < 1) return -1;
    const int P = (Sk + num_splits - 1) / num_splits; /* keys per partition */
    for (int s = 0; s < num_splits; ++s) {
        const int lo = s * P;
        const int hi = (lo + P < Sk) ? lo + P : Sk;
        double *os = o_part + (size_t)s * D;
        for (int d = 0; d < D; ++d) os[d] = 0.0;
        if (lo >= hi) { m_part[s] = -INFINITY; l_part[s] = 0.0; continue; }

        double m = -INFINITY;
        for (int j = lo; j < hi; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q[d] * k[(size_t)j * D + d];
            if (scale * dot > m) m = scale * dot;
        }
        double l = 0.0;
        for (int j = lo; j < hi; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q[d] * k[(size_t)j * D + d];
            const double p = exp(scale * dot - m);
            l += p;
            for (int d = 0; d < D; ++d) os[d] += p * v[(size_t)j * D + d];
        }
        m_part[s] = m;
        l_part[s] = l;
    }
    return 0;
}

/* ---- split-K decoding, phase 2 ------------------------------------------- */

/* One head. Inputs from phase 1; o: [D], lse: scalar. */
int oracle_splitkv_merge(const double *o_part, const double *m_part, const double *l_part,
                         int num_splits, int D, double *o, double *lse)
{
    if (num_splits < 1 || D < 1) return -1;
    double mg = -INFINITY;
    for (int s = 0; s < num_splits; ++s)
        if (m_part[s] > mg) mg = m_part[s];
    if (mg == -INFINITY) return -1; /* every partition empty: nothing to merge */
    double lg = 0.0;
    for (int s = 0; s < num_splits; ++s) lg += exp(m_part[s] - mg) * l_part[s];
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int s = 0; s < num_splits; ++s)
            acc += exp(m_part[s] - mg) / lg * o_part[(size_t)s * D + d];
        o[d] = acc;
    }
    *lse = mg + log(lg);
    return 0;
}

/* ---- backward pass ------------------------------------------------------ */

/* One head. q, dout: [Sq][D]; k, v: [Sk][D]. Outputs dq: [Sq][D],
 * dk and dv: [Sk][D]. */
int oracle_attention_bwd_head(const double *q, const double *k, const double *v,
                              const double *dout, int Sq, int Sk, int D, int causal,
                              double scale, double *dq, double *dk, double *dv)
{
    if (Sq < 1 || Sk < 1 || D < 1) return -1;
    double *P = (double *)malloc((size_t)Sq * (size_t)Sk * sizeof(double));
    double *dS = (double *)malloc((size_t)Sq * (size_t)Sk * sizeof(double));
    double *o = (double *)malloc((size_t)D * sizeof(double));
    if (!P || !dS || !o) { free(P); free(dS); free(o); return -2; }

    for (int i = 0; i < Sq; ++i) {
        double *Pi = P + (size_t)i * Sk;
        /* S_ij = scale * q_i . k_j, masked; P_i = softmax(S_i) */
        double m = -INFINITY;
        for (int j = 0; j < Sk; ++j) {
            double qk = 0.0;
            for (int d = 0; d < D; ++d) qk += q[(size_t)i * D + d] * k[(size_t)j * D + d];
            Pi[j] = (causal && j > i) ? -INFINITY : scale * qk;
            if (Pi[j] > m) m = Pi[j];
        }
        double l = 0.0;
        for (int j = 0; j < Sk; ++j) {
            Pi[j] = exp(Pi[j] - m);
            l += Pi[j];
        }
        for (int j = 0; j < Sk; ++j) Pi[j] /= l;
        /* O_i = sum_j P_ij v_j, then D_i = sum_k dO_ik O_ik */
        double Di = 0.0;
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int j = 0; j < Sk; ++j) acc += Pi[j] * v[(size_t)j * D + d];
            o[d] = acc;
            Di += dout[(size_t)i * D + d] * acc;
        }
        /* dP_ij = dO_i . v_j, dS_ij = P_ij (dP_ij - D_i) */
        for (int j = 0; j < Sk; ++j) {
            double dp = 0.0;
            for (int d = 0; d < D; ++d) dp += dout[(size_t)i * D + d] * v[(size_t)j * D + d];
            dS[(size_t)i * Sk + j] = Pi[j] * (dp - Di);
        }
    }
    /* dQ_i = scale * sum_j dS_ij k_j */
    for (int i = 0; i < Sq; ++i)
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int j = 0; j < Sk; ++j) acc += dS[(size_t)i * Sk + j] * k[(size_t)j * D + d];
            dq[(size_t)i * D + d] = scale * acc;
        }
    /* dK_j = scale * sum_i dS_ij q_i, dV_j = sum_i P_ij dO_i (summed over i
     * in the outer loop so that P and dS are read row by row) */
    for (size_t x = 0; x < (size_t)Sk * D; ++x) { dk[x] = 0.0; dv[x] = 0.0; }
    for (int i = 0; i < Sq; ++i)
        for (int j = 0; j < Sk; ++j) {
            const double ds_ij = dS[(size_t)i * Sk + j], p_ij = P[(size_t)i * Sk + j];
            for (int d = 0; d < D; ++d) {
                dk[(size_t)j * D + d] += ds_ij * q[(size_t)i * D + d];
                dv[(size_t)j * D + d] += p_ij * dout[(size_t)i * D + d];
            }
        }
    for (size_t x = 0; x < (size_t)Sk * D; ++x) dk[x] *= scale;
    free(P);
    free(dS);
    free(o);
    return 0;
}

typedef struct {
    const double *q, *k, *v, *dout;
    double *dq, *dk, *dv;
    int Sq, Sk, D, causal;
    double scale;
    int head_begin, head_end;
    int status;
} bwd_job;

static void *run_bwd_heads(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    jb->status = 0;
    for (int h = jb->head_begin; h < jb->head_end && jb->status == 0; ++h) {
        const size_t qo = (size_t)h * jb->Sq * jb->D, ko = (size_t)h * jb->Sk * jb->D;
        jb->status = oracle_attention_bwd_head(jb->q + qo, jb->k + ko, jb->v + ko, jb->dout + qo,
                                               jb->Sq, jb->Sk, jb->D, jb->causal, jb->scale,
                                               jb->dq + qo, jb->dk + ko, jb->dv + ko);
    }
    return NULL;
}

/* q, dout, dq: [BH][Sq][D]; k, v, dk, dv: [BH][Sk][D]. */
int oracle_attention_bwd(const double *q, const double *k, const double *v, const double *dout,
                         double *dq, double *dk, double *dv, int BH, int Sq, int Sk, int D,
                         int causal, double scale, int nthreads)
{
    if (BH < 0) return -1;
    if (BH == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > BH) nthreads = BH;
    bwd_job *jobs = (bwd_job *)calloc((size_t)nthreads, sizeof(bwd_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -2; }
    for (int t = 0; t < nthreads; ++t) {
        bwd_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->dout = dout;
        jb->dq = dq; jb->dk = dk; jb->dv = dv;
        jb->Sq = Sq; jb->Sk = Sk; jb->D = D; jb->causal = causal; jb->scale = scale;
        jb->head_begin = (int)((long long)BH * t / nthreads);
        jb->head_end = (int)((long long)BH * (t + 1) / nthreads);
    }
    int status = 0, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, run_bwd_heads, &jobs[t]) != 0) { status = -2; break; }
        ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    for (int t = 0; t < started && status == 0; ++t) status = jobs[t].status;
    free(jobs);
    free(tids);
    return status;
}

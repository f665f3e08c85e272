/*
 * maxsim_oracle.c -- fp64 CPU oracle for the late-interaction MaxSim operator.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the package smoke check and the CPU-baseline leg of the benchmark may load
 * it.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (Late Interaction Kernels README, "What does it compute?"):
 *
 *     MaxSim(Q, D) = sum over valid query tokens i of
 *                    max over valid document tokens j of  Q_i . D_j
 *
 * Mask and sentinel rules (same README, "Scoring interface"):
 *   - a query mask removes token i from the sum;
 *   - a document mask removes token j from the max;
 *   - a NULL mask means every token is valid;
 *   - a document with no valid token scores -1e9 (a fixed value, whatever
 *     the query), and no query token has an argmax for it (-1).
 *   - a non-empty document scored against a query with no valid token
 *     scores exactly 0 (an empty sum).
 *
 * Exactness (LIK announcement thread, post 5/N: identical to the naive
 * computation, no approximation): every similarity is a plain dot product
 * summed in fp64 over ascending k; the max keeps the FIRST (lowest j) token
 * that reaches it, because the running max only moves on a strictly larger
 * value; the score sums the maxima in fp64 over ascending i.
 *
 * Layouts (README, "Scoring interface" table; colpali PR "Add support for
 * late-interaction-kernels (LIK)", Design section, for the per-query
 * candidate layout):
 *   all-pairs  Q[Nq,Lq,dim] x D[Nd,Ld,dim]   -> scores[Nq,Nd], argmax[Nq,Nd,Lq]
 *   pairwise   Q[B,Lq,dim]  x D[B,Ld,dim]    -> scores[B],     argmax[B,Lq]
 *   kd         Q[B,Lq,dim]  x D[B,N,Ld,dim]  -> scores[B,N],   argmax[B,N,Lq]
 *
 * Backward (README, "What does it compute?": gradients flow into query and
 * document embeddings; LIK thread post 5/N: the backward is fused).  The
 * score is piecewise linear in Q and D: for each valid i of a non-empty
 * document the only active term is Q_i . D_a with a = argmax, so
 *     dScore/dQ_i = D_a          and          dScore/dD_a += Q_i .
 * With upstream gradient g per score the oracle accumulates
 *     gQ[q,i] += g * D[d,a]    and    gD[d,a] += g * Q[q,i]
 * in fp64, reading the argmax that its own forward saved.
 *
 * Inputs arrive in their storage type (f32, f16, bf16 or f64) and are widened
 * exactly to fp64 before any arithmetic, so the oracle sees the same
 * dtype-rounded values as the GPU.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_F64 = 3 };

#define ORACLE_EMPTY_DOC_SCORE (-1e9)

/* ---- exact widening of one stored element to fp64 -------------------- */

static double widen_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double widen_bf16(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16; /* bf16 is the top half of an f32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double widen(const void* base, int dtype, int64_t idx)
{
    switch (dtype) {
    case ORACLE_F32: return (double)((const float*)base)[idx];
    case ORACLE_F16: return widen_f16(((const uint16_t*)base)[idx]);
    case ORACLE_BF16: return widen_bf16(((const uint16_t*)base)[idx]);
    default: return ((const double*)base)[idx];
    }
}

/* Widen n consecutive elements starting at element offset off. */
static double* widen_block(const void* base, int dtype, int64_t off, int64_t n)
{
    double* out = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!out) return NULL;
    for (int64_t t = 0; t < n; ++t) out[t] = widen(base, dtype, off + t);
    return out;
}

/* ---- one query against one document ---------------------------------- */

/*
 * q: [Lq,dim] fp64, d: [Ld,dim] fp64; qm/dm: 1 byte per token (0 = padding)
 * or NULL.  Writes argmax[i] (or -1) and, when gap != NULL, the distance
 * between the best and second-best valid similarity of token i (+inf when
 * only one document token is valid, NaN where there is no argmax).
 * Returns the score.
 */
double oracle_pair(const double* q, const uint8_t* qm, int64_t Lq,
                   const double* d, const uint8_t* dm, int64_t Ld, int64_t dim,
                   int32_t* argmax, double* gap)
{
    int any_valid_doc_token = 0;
    for (int64_t j = 0; j < Ld; ++j)
        if (!dm || dm[j]) any_valid_doc_token = 1;

    if (!any_valid_doc_token) {
        for (int64_t i = 0; i < Lq; ++i) {
            if (argmax) argmax[i] = -1;
            if (gap) gap[i] = NAN;
        }
        return ORACLE_EMPTY_DOC_SCORE;
    }

    double score = 0.0;
    for (int64_t i = 0; i < Lq; ++i) {
        if (qm && !qm[i]) {
            if (argmax) argmax[i] = -1;
            if (gap) gap[i] = NAN;
            continue;
        }
        double best = -INFINITY, second = -INFINITY;
        int32_t best_j = -1;
        for (int64_t j = 0; j < Ld; ++j) {
            if (dm && !dm[j]) continue;
            double s = 0.0;
            for (int64_t k = 0; k < dim; ++k) s += q[i * dim + k] * d[j * dim + k];
            if (s > best) {
                second = best;
                best = s;
                best_j = (int32_t)j;
            } else if (s > second) {
                second = s;
            }
        }
        score += best;
        if (argmax) argmax[i] = best_j;
        if (gap) gap[i] = best - second;
    }
    return score;
}

/* Score query qidx of Q against document didx of D (both in token-block units). */
static double score_blocks(const void* Q, const void* D, int dtype,
                           int64_t qidx, int64_t didx, int64_t Lq, int64_t Ld, int64_t dim,
                           const uint8_t* qmask, const uint8_t* dmask,
                           int32_t* argmax, double* gap)
{
    double* q = widen_block(Q, dtype, qidx * Lq * dim, Lq * dim);
    double* d = widen_block(D, dtype, didx * Ld * dim, Ld * dim);
    double s = NAN;
    if (q && d)
        s = oracle_pair(q, qmask ? qmask + qidx * Lq : NULL, Lq,
                        d, dmask ? dmask + didx * Ld : NULL, Ld, dim, argmax, gap);
    free(q);
    free(d);
    return s;
}

/* ---- forward, one function per layout --------------------------------- */

/*
 * Every (query, document) pair of a layout is independent; OpenMP spreads the
 * pairs over the host cores.  argmax and gap may be NULL.
 */
void oracle_allpairs_fwd(const void* Q, const void* D, int dtype,
                         int64_t Nq, int64_t Nd, int64_t Lq, int64_t Ld, int64_t dim,
                         const uint8_t* qmask, const uint8_t* dmask,
                         double* scores, int32_t* argmax, double* gap)
{
    int64_t pairs = Nq * Nd;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < pairs; ++p) {
        int64_t qi = p / Nd, di = p % Nd;
        scores[p] = score_blocks(Q, D, dtype, qi, di, Lq, Ld, dim, qmask, dmask,
                                 argmax ? argmax + p * Lq : NULL, gap ? gap + p * Lq : NULL);
    }
}

/* Pair b scores query b against document b only. */
void oracle_pairwise_fwd(const void* Q, const void* D, int dtype,
                         int64_t B, int64_t Lq, int64_t Ld, int64_t dim,
                         const uint8_t* qmask, const uint8_t* dmask,
                         double* scores, int32_t* argmax, double* gap)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t b = 0; b < B; ++b)
        scores[b] = score_blocks(Q, D, dtype, b, b, Lq, Ld, dim, qmask, dmask,
                                 argmax ? argmax + b * Lq : NULL, gap ? gap + b * Lq : NULL);
}

/* Query b scores its own N candidates D[b,0..N-1]; candidate (b,n) is document b*N+n. */
void oracle_kd_fwd(const void* Q, const void* D, int dtype,
                   int64_t B, int64_t N, int64_t Lq, int64_t Ld, int64_t dim,
                   const uint8_t* qmask, const uint8_t* dmask,
                   double* scores, int32_t* argmax, double* gap)
{
    int64_t pairs = B * N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < pairs; ++p) {
        int64_t b = p / N;
        scores[p] = score_blocks(Q, D, dtype, b, p, Lq, Ld, dim, qmask, dmask,
                                 argmax ? argmax + p * Lq : NULL, gap ? gap + p * Lq : NULL);
    }
}

/* ---- backward ---------------------------------------------------------- */

/*
 * Generic backward over a list of (query, document) pairs: pair p joins
 * query qidx[p] with document didx[p], has upstream gradient g[p] and saved
 * argmax argmax[p*Lq .. p*Lq+Lq-1].  gQ [nQ,Lq,dim] and gD [nD,Ld,dim] are
 * overwritten.  gQ rows are owned by their query and gD rows by their
 * document, so each parallel loop writes disjoint rows.
 */
static void backward_pairs(const void* Q, const void* D, int dtype,
                           int64_t nQ, int64_t nD, int64_t npairs,
                           const int64_t* qidx, const int64_t* didx,
                           int64_t Lq, int64_t Ld, int64_t dim,
                           const double* g, const int32_t* argmax,
                           double* gQ, double* gD)
{
    if (gQ) {
        memset(gQ, 0, (size_t)(nQ * Lq * dim) * sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t qq = 0; qq < nQ; ++qq)
            for (int64_t p = 0; p < npairs; ++p) {
                if (qidx[p] != qq) continue;
                for (int64_t i = 0; i < Lq; ++i) {
                    int32_t a = argmax[p * Lq + i];
                    if (a < 0) continue;
                    for (int64_t k = 0; k < dim; ++k)
                        gQ[(qq * Lq + i) * dim + k] +=
                            g[p] * widen(D, dtype, (didx[p] * Ld + a) * dim + k);
                }
            }
    }
    if (gD) {
        memset(gD, 0, (size_t)(nD * Ld * dim) * sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t dd = 0; dd < nD; ++dd)
            for (int64_t p = 0; p < npairs; ++p) {
                if (didx[p] != dd) continue;
                for (int64_t i = 0; i < Lq; ++i) {
                    int32_t a = argmax[p * Lq + i];
                    if (a < 0) continue;
                    for (int64_t k = 0; k < dim; ++k)
                        gD[(dd * Ld + a) * dim + k] +=
                            g[p] * widen(Q, dtype, (qidx[p] * Lq + i) * dim + k);
                }
            }
    }
}

static int64_t* index_array(int64_t n)
{
    return (int64_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
}

void oracle_allpairs_bwd(const void* Q, const void* D, int dtype,
                         int64_t Nq, int64_t Nd, int64_t Lq, int64_t Ld, int64_t dim,
                         const double* grad_out, const int32_t* argmax,
                         double* gQ, double* gD)
{
    int64_t n = Nq * Nd;
    int64_t *qi = index_array(n), *di = index_array(n);
    for (int64_t p = 0; p < n; ++p) {
        qi[p] = p / Nd;
        di[p] = p % Nd;
    }
    backward_pairs(Q, D, dtype, Nq, Nd, n, qi, di, Lq, Ld, dim, grad_out, argmax, gQ, gD);
    free(qi);
    free(di);
}

void oracle_pairwise_bwd(const void* Q, const void* D, int dtype,
                         int64_t B, int64_t Lq, int64_t Ld, int64_t dim,
                         const double* grad_out, const int32_t* argmax,
                         double* gQ, double* gD)
{
    int64_t *qi = index_array(B), *di = index_array(B);
    for (int64_t p = 0; p < B; ++p) qi[p] = di[p] = p;
    backward_pairs(Q, D, dtype, B, B, B, qi, di, Lq, Ld, dim, grad_out, argmax, gQ, gD);
    free(qi);
    free(di);
}

void oracle_kd_bwd(const void* Q, const void* D, int dtype,
                   int64_t B, int64_t N, int64_t Lq, int64_t Ld, int64_t dim,
                   const double* grad_out, const int32_t* argmax,
                   double* gQ, double* gD)
{
    int64_t n = B * N;
    int64_t *qi = index_array(n), *di = index_array(n);
    for (int64_t p = 0; p < n; ++p) {
        qi[p] = p / N;
        di[p] = p;
    }
    backward_pairs(Q, D, dtype, B, n, n, qi, di, Lq, Ld, dim, grad_out, argmax, gQ, gD);
    free(qi);
    free(di);
}

/*
 * Cross-entropy head over score rows (colpali PR "Add support for
 * late-interaction-kernels (LIK)", "What this PR adds": the in-batch ColBERT
 * losses score a query against the batch's documents with its own document
 * as the target, the negative-document losses score it against its own
 * candidates with the positive first; "Results": the benchmarks time that
 * head, forward and backward).  For every row r of scores[rows, cols] with
 * logits z = scale * scores[r, :] and target t = target[r]:
 *     row_loss[r] = log(sum over c of exp(z_c)) - z_t
 *     grad[r, c]  = scale * (exp(z_c) / sum exp(z) - [c == t]) / rows
 * and loss = (sum over r of row_loss[r]) / rows, i.e. the mean cross-entropy
 * and its gradient with respect to the scores.  The log-sum-exp subtracts
 * the row max first; everything is fp64.  A row whose target is outside
 * [0, cols) gets row_loss 0 and a zero gradient and still counts in the mean.
 */
void oracle_ce_rows(const double* scores, int64_t rows, int64_t cols, const int32_t* target,
                    double scale, double* row_loss, double* grad, double* loss)
{
    double total = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        const double* s = scores + r * cols;
        double* gr = grad + r * cols;
        const int32_t t = target[r];
        if (t < 0 || t >= cols) {
            row_loss[r] = 0.0;
            for (int64_t c = 0; c < cols; ++c) gr[c] = 0.0;
            continue;
        }
        double m = -INFINITY;
        for (int64_t c = 0; c < cols; ++c)
            if (scale * s[c] > m) m = scale * s[c];
        double sum = 0.0;
        for (int64_t c = 0; c < cols; ++c) sum += exp(scale * s[c] - m);
        const double lse = m + log(sum);
        row_loss[r] = lse - scale * s[t];
        for (int64_t c = 0; c < cols; ++c)
            gr[c] = scale * (exp(scale * s[c] - lse) - (c == t ? 1.0 : 0.0)) / (double)rows;
        total += row_loss[r];
    }
    *loss = rows > 0 ? total / (double)rows : 0.0;
}

/* Number of threads the OpenMP loops above use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the number of threads for later calls (n <= 0 leaves it unchanged). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

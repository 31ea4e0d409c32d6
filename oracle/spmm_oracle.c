/*
 * CPU oracle for CSR SpMM -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark load this file's library. The product path (the CUDA library)
 * never calls it and shares no code, header or constant with it.
 *
 * What it computes (graph-spmm model card, "API" and "Correctness"; ParamSpMM
 * section 2 "Background", Algorithm 1; GE-SpMM section V-A on general
 * SpMM-like reductions):
 *
 *   A is M x K in CSR: row i holds the stored entries p in
 *   [rowptr[i], rowptr[i+1]) with column col[p] and value a_p = val[p]
 *   (a_p = 1 for every entry when val is NULL, an unweighted adjacency).
 *   B is K x N, row-major. For every output element (i, k) and every stored
 *   entry p of row i, taken in CSR order, x_p = a_p * B[col[p], k].
 *
 *   sum : C[i,k] = sum_p x_p.  The products of two fp32 numbers are exact in
 *         fp64, the running sum is fp64, and the result is rounded to fp32 once.
 *         Duplicate (row, col) entries each contribute (model card,
 *         "Correctness": a real CSR may hold duplicate pairs and they are summed).
 *   mean: C[i,k] = (sum_p x_p) / d_i with d_i = rowptr[i+1] - rowptr[i], the
 *         number of stored entries, divided in fp64 and rounded once; an empty
 *         row gives 0 (model card, "API": empty rows are 0).
 *   max : candidates y_p = fl32(x_p), the fp32-rounded product (the fp64
 *         product is exact, so this is the correctly rounded fp32 product).
 *         (y, j) beats (y*, j*) when y > y*, or y == y* and j < j*: ties go to
 *         the smallest column index, and -0 == +0. The first entry seeds the
 *         running best. C[i,k] = y*, argmax[i,k] = j*; an empty row gives
 *         (0, -1) (model card, "API": spmm_max returns (values, argmax),
 *         empty rows are (0, -1)).
 *
 *   T[i,k] = sum_p |x_p| is returned beside sum/mean as the scale of the
 *   floating-point tolerance |err| <= 1e-5 * T + 1e-6.
 *
 * Epilogue (a GCN layer's aggregation followed by its node update, "Dual-Metric
 * Partitioning with Adaptive Kernel Execution for Efficient GCN Acceleration",
 * introduction; here the bias and activation of that update):
 *   with a bias vector b [N] and/or ReLU, the output is
 *   act(R[i,k] + b[k]) where R is the value defined above before its final
 *   rounding (the fp64 sum, or the fp64 mean, or the fp32 max), the addition
 *   is done in fp64 and rounded to fp32 once, and ReLU(x) = x > 0 ? x : +0 is
 *   applied last. An empty row has R = 0. argmax is not affected.
 *
 * Descriptors (RA-SpMM abstract and "routing rules": one O(M) pass over the
 * row pointers gives M, the mean row degree and the coefficient of variation
 * of the row degree): dbar = nnz / M and CV_d = std(d) / mean(d), std taken
 * over all M rows (empty rows included) with divisor M.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC. Rows are
 * independent and each is reduced by one thread in CSR order, so the result
 * does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_SUM = 0, ORACLE_MEAN = 1, ORACLE_MAX = 2 };
enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1 };

/* Mutation switch for the pin tests only: a build with -DORACLE_PLANT=n plants
 * one known mistake so the tests can show that their pins reject it.
 * 0 (the default) is the oracle as specified above. */
#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

typedef struct {
    int64_t M, nnz, d_max, n_empty;
    double dbar, cv;
} oracle_desc;

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* The epilogue on one value r (fp64): add the bias, round once, then ReLU. */
static float oracle_epilogue(double r, const float *bias, int64_t k, int act) {
#if ORACLE_PLANT == 6
    if (act == ORACLE_ACT_RELU) r = r > 0.0 ? r : 0.0;   /* planted: ReLU before the bias */
    return (float)(bias ? r + (double)bias[k] : r);
#else
    float c = (float)(bias ? r + (double)bias[k] : r);
    if (act == ORACLE_ACT_RELU) c = c > 0.0f ? c : 0.0f;
    return c;
#endif
}

/* One output row. S and Tacc are caller scratch of N doubles each. */
static void oracle_row(int64_t i, int64_t K, int64_t N, const int32_t *rowptr, const int32_t *col,
                       const float *val, const float *B, int reduce, const float *bias, int act,
                       float *Crow, int32_t *Arow, float *Trow, double *S, double *Tacc) {
    const int64_t p0 = rowptr[i], p1 = rowptr[i + 1];
    const int64_t d = p1 - p0;
    if (reduce == ORACLE_MAX) {
        if (d == 0) {
            for (int64_t k = 0; k < N; ++k) {
                Crow[k] = oracle_epilogue(0.0, bias, k, act);
                if (Arow) Arow[k] = -1;
            }
            return;
        }
        /* seed with the first entry */
        {
            const int32_t j = col[p0];
            const double a = val ? (double)val[p0] : 1.0;
            for (int64_t k = 0; k < N; ++k) {
                Crow[k] = (float)(a * (double)B[(int64_t)j * N + k]);
                if (Arow) Arow[k] = j;
            }
        }
        int32_t *best_j = Arow;
        int32_t *tmp = NULL;
        if (!best_j) {
            tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
            for (int64_t k = 0; k < N; ++k) tmp[k] = col[p0];
            best_j = tmp;
        }
        for (int64_t p = p0 + 1; p < p1; ++p) {
            const int32_t j = col[p];
            const double a = val ? (double)val[p] : 1.0;
            const float *Bj = B + (int64_t)j * N;
            for (int64_t k = 0; k < N; ++k) {
                const float y = (float)(a * (double)Bj[k]);
#if ORACLE_PLANT == 4
                if (y > Crow[k] || (y == Crow[k] && j > best_j[k])) {
#else
                if (y > Crow[k] || (y == Crow[k] && j < best_j[k])) {
#endif
                    Crow[k] = y;
                    best_j[k] = j;
                }
            }
        }
        free(tmp);
        if (bias || act != ORACLE_ACT_NONE)
            for (int64_t k = 0; k < N; ++k) Crow[k] = oracle_epilogue((double)Crow[k], bias, k, act);
        return;
    }
    for (int64_t k = 0; k < N; ++k) {
        S[k] = 0.0;
        Tacc[k] = 0.0;
    }
    for (int64_t p = p0; p < p1; ++p) {
#if ORACLE_PLANT == 1
        if (p == p1 - 1) break;                       /* planted: drops a term */
#endif
        int32_t j = col[p];
#if ORACLE_PLANT == 2
        j = (int32_t)((j + 1) % K);                   /* planted: wrong index */
#endif
        const double a = val ? (double)val[p] : 1.0;
        const float *Bj = B + (int64_t)j * N;
        for (int64_t k = 0; k < N; ++k) {
#if ORACLE_PLANT == 3
            const double x = a * (double)B[((int64_t)k % K) * N + (j % N)]; /* planted: transposed */
#else
            const double x = a * (double)Bj[k];
#endif
            S[k] += x;
            Tacc[k] += fabs(x);
        }
    }
    for (int64_t k = 0; k < N; ++k) {
        double r;
        if (reduce == ORACLE_MEAN)
#if ORACLE_PLANT == 5
            r = d ? S[k] / (double)(d + 1) : 0.0;  /* planted: wrong divisor */
#else
            r = d ? S[k] / (double)d : 0.0;
#endif
        else
            r = S[k];
        Crow[k] = oracle_epilogue(r, bias, k, act);
        if (Trow) Trow[k] = (float)Tacc[k];
    }
}

/* Rows given by `rows` (nrows of them; NULL means rows 0..M-1 in order).
 * Output row r of C / argmax / T corresponds to input row rows[r].
 * Returns 0, or -1 on a bad argument (the caller sees it as an exception). */
int oracle_spmm_rows_ex(int64_t M, int64_t K, int64_t N, const int32_t *rowptr,
                        const int32_t *col, const float *val, const float *B, int reduce,
                        const float *bias, int act, const int64_t *rows, int64_t nrows, float *C,
                        int32_t *argmax, float *T) {
    if (M < 0 || K < 0 || N < 0 || nrows < 0 || !rowptr || !C) return -1;
    if (reduce < ORACLE_SUM || reduce > ORACLE_MAX) return -1;
    if (act != ORACLE_ACT_NONE && act != ORACLE_ACT_RELU) return -1;
    if (rows) {
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= M) return -1;
    }
    int bad = 0;
#pragma omp parallel reduction(| : bad)
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        double *Tacc = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!S || !Tacc) bad = 1;
#pragma omp for schedule(dynamic, 256)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!S || !Tacc) continue;
            const int64_t i = rows ? rows[r] : r;
            oracle_row(i, K, N, rowptr, col, val, B, reduce, bias, act, C + r * N,
                       argmax ? argmax + r * N : NULL, T ? T + r * N : NULL, S, Tacc);
        }
        free(S);
        free(Tacc);
    }
    return bad ? -1 : 0;
}

int oracle_spmm_rows(int64_t M, int64_t K, int64_t N, const int32_t *rowptr,
                     const int32_t *col, const float *val, const float *B, int reduce,
                     const int64_t *rows, int64_t nrows, float *C, int32_t *argmax, float *T) {
    return oracle_spmm_rows_ex(M, K, N, rowptr, col, val, B, reduce, NULL, ORACLE_ACT_NONE, rows,
                               nrows, C, argmax, T);
}

int oracle_spmm(int64_t M, int64_t K, int64_t N, const int32_t *rowptr, const int32_t *col,
                const float *val, const float *B, int reduce, float *C, int32_t *argmax,
                float *T) {
    return oracle_spmm_rows(M, K, N, rowptr, col, val, B, reduce, NULL, M, C, argmax, T);
}

/* Degree descriptors over all M rows, integer sums exact in 64 bits. */
int oracle_descriptors(int64_t M, const int32_t *rowptr, oracle_desc *out) {
    if (M < 0 || !out || (M > 0 && !rowptr)) return -1;
    memset(out, 0, sizeof(*out));
    out->M = M;
    if (M == 0) return 0;
    uint64_t s1 = 0, s2 = 0;
    int64_t dmax = 0, empty = 0;
    for (int64_t i = 0; i < M; ++i) {
        const int64_t d = (int64_t)rowptr[i + 1] - (int64_t)rowptr[i];
        if (d < 0) return -1;
        s1 += (uint64_t)d;
        s2 += (uint64_t)d * (uint64_t)d;
        if (d > dmax) dmax = d;
        if (d == 0) ++empty;
    }
    out->nnz = (int64_t)s1;
    out->d_max = dmax;
    out->n_empty = empty;
    out->dbar = (double)s1 / (double)M;
    const double var = (double)s2 / (double)M - out->dbar * out->dbar;
    out->cv = (s1 == 0) ? 0.0 : sqrt(var > 0.0 ? var : 0.0) / out->dbar;
    return 0;
}

/* ------------------------------------------------------------------------
 * Backward of the three reductions (graph-spmm card, "Requirements and
 * limits": the backward of a sum aggregation is the transposed product,
 * from a second adjacency on the reversed edge list; "Method"/"API": the
 * argmax returned by spmm_max feeds the max-pool backward).
 *
 * oracle_transpose: A^T in CSR. Row j of A^T holds every stored entry (i, j)
 * of A, in increasing i, and entries of one row i in their CSR order (a
 * stable counting sort of the entries by column). With scale_mean, the value
 * of entry (i, j) is a_ij / d_i rounded once (1 / d_i for an unweighted A):
 * then A_mean^T . dC is the mean's backward.
 *
 * oracle_maxpool_backward: the derivative of the max reduction with respect
 * to B. The forward value C[i, k] is the product y_p = fl32(a_p * B[j_p, k])
 * of ONE stored entry p of row i (duplicates are legal CSR, graph-spmm card,
 * "Correctness"), so only that entry passes the gradient:
 *   dB[j, k] = sum over rows i with argmax[i, k] == j of a_w * dC[i, k],
 * where w is the winning copy of column j in row i: among the stored entries p
 * of row i with col[p] == j, the one with the largest y_p, the smallest
 * storage position on equal y_p (fp64 sum, rounded once). Without duplicated
 * pairs w is the only entry of column j in the row.
 * ------------------------------------------------------------------------ */
int oracle_transpose(int64_t M, int64_t K, const int32_t *rowptr, const int32_t *col,
                     const float *val, int scale_mean, int32_t *rowptrT, int32_t *colT,
                     float *valT) {
    if (M < 0 || K < 0 || !rowptr || !rowptrT) return -1;
    const int64_t nnz = rowptr[M];
    for (int64_t j = 0; j <= K; ++j) rowptrT[j] = 0;
    for (int64_t p = 0; p < nnz; ++p) {
        if (col[p] < 0 || col[p] >= K) return -1;
        rowptrT[col[p] + 1] += 1;
    }
    for (int64_t j = 0; j < K; ++j) rowptrT[j + 1] += rowptrT[j];
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
    if (!next) return -1;
    for (int64_t j = 0; j < K; ++j) next[j] = rowptrT[j];
    for (int64_t i = 0; i < M; ++i) {
        const int64_t d = rowptr[i + 1] - rowptr[i];
        for (int64_t p = rowptr[i]; p < rowptr[i + 1]; ++p) {
            const int32_t q = next[col[p]]++;
            colT[q] = (int32_t)i;
            if (valT) {
                const double a = val ? (double)val[p] : 1.0;
                valT[q] = scale_mean ? (float)(a / (double)d) : (float)a;
            }
        }
    }
    free(next);
    return 0;
}

int oracle_maxpool_backward(int64_t M, int64_t K, int64_t N, const int32_t *rowptr,
                            const int32_t *col, const float *val, const float *B,
                            const int32_t *argmax, const float *dC, float *dB) {
    if (M < 0 || K < 0 || N < 0 || !rowptr || !argmax || !dC || !dB) return -1;
    if (val && !B && rowptr[M] > 0) return -1;
    double *acc = (double *)calloc((size_t)(K * N > 0 ? K * N : 1), sizeof(double));
    if (!acc) return -1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t k = 0; k < N; ++k) {
            const int32_t j = argmax[i * N + k];
            if (j < 0) continue;                      /* empty row: no gradient */
            if (j >= K) { free(acc); return -1; }
            /* the winning copy of column j: largest fp32 product, first on ties */
            int64_t w = -1;
            float y_w = 0.0f;
            for (int64_t p = rowptr[i]; p < rowptr[i + 1]; ++p) {
                if (col[p] != j) continue;
                const float a = val ? val[p] : 1.0f;
                const float y = val ? (float)((double)a * (double)B[(int64_t)j * N + k]) : 0.0f;
                if (w < 0 || y > y_w) { w = p; y_w = y; }
            }
            if (w < 0) { free(acc); return -1; }      /* argmax names no stored column */
            const double a_w = val ? (double)val[w] : 1.0;
            acc[(int64_t)j * N + k] += a_w * (double)dC[i * N + k];
        }
    }
    for (int64_t q = 0; q < K * N; ++q) dB[q] = (float)acc[q];
    free(acc);
    return 0;
}

/*
 * oracle.c -- slow, plain FP64 CPU reference for the row-major FP32 GEMM family.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA library is
 * compared against.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load it.  It shares no code, header or table with
 * the CUDA path, and the CUDA path never calls it.
 *
 * What it computes (one output element at a time, exactly the definition):
 *
 *   GEMM 优化详解, "GEMM 基础理论 / 数学定义":   C = alpha * A x B + beta * C,
 *       A is M x K, B is K x N, C is M x N.
 *   第5章-基础Kernel, "1.1 什么是矩阵乘法":       C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *       (0-based k, row-major storage, A[i*K + k] indexing as in "2. Naive 矩阵乘法实现").
 *   GEMM 优化详解, "Level 6: Kernel Fusion":      the fused layer adds bias[col] to every
 *       element of column col and then applies ReLU(x) = max(0, x).  Reading for the
 *       row-broadcast variant of that epilogue: row_bias[row] is added to every element
 *       of row row, in the same place as bias[col].
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - op(A) / op(B) with BLAS-style row-major transposes and leading dimensions:
 *       op(A)(i,k) = ta ? A[k*lda + i] : A[i*lda + k]
 *       op(B)(k,j) = tb ? B[j*ldb + k] : B[k*ldb + j]
 *   - beta == 0: C0 is not read (it may hold NaN or be NULL).
 *   - alpha == 0 or K == 0: the product term is not formed and A, B are not read.
 *   - the fused order is relu(alpha*sum + beta*C0 + bias[j] + row_bias[i]); ReLU maps
 *     NaN to 0 (the page's fmaxf(0, val)).
 *
 * Arithmetic: every product of two floats is exact in double (24+24 < 53 bits),
 * the k-sum runs in ascending k exactly as written in the definition, and the
 * epilogue is evaluated in double.  The file must be compiled with
 * -ffp-contract=off so that no fused multiply-add changes the rounding between
 * machines.
 *
 * Besides the value it returns, per element,
 *     mag(i,j) = |alpha| * sum_k |op(A)(i,k)| * |op(B)(k,j)| + |beta| * |C0(i,j)| + |bias[j]|
 *                + |row_bias[i]|
 * which scales the per-element acceptance bound of the tests.
 *
 * Rows of the output are split over POSIX threads; the thread count is an
 * argument so the same code can be timed on one core or on all of them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

typedef struct {
    int ta, tb;
    int64_t M, N, K;
    double alpha, beta;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    const float *C0;
    int64_t ldc;
    const float *bias;     /* length N, per column, or NULL */
    const float *row_bias; /* length M, per row, or NULL */
    int relu;
    const int64_t *rows; /* NULL: all M rows */
    int64_t nrows;
    double *out; /* nrows x N, dense (row stride N) */
    double *mag; /* nrows x N, dense, may be NULL */
    int64_t first, last; /* this worker's slice of [0, nrows) */
    int status;
} job_t;

static double a_at(const job_t *j, int64_t i, int64_t k)
{
    return (double)(j->ta ? j->A[k * j->lda + i] : j->A[i * j->lda + k]);
}

static double b_at(const job_t *j, int64_t k, int64_t c)
{
    return (double)(j->tb ? j->B[c * j->ldb + k] : j->B[k * j->ldb + c]);
}

/* One output row i: out[c] = epilogue(sum_k op(A)(i,k) * op(B)(k,c)). */
static void one_row(const job_t *j, int64_t i, double *orow, double *mrow, double *arow)
{
    const int64_t N = j->N, K = j->K;
    const int products = (K > 0 && j->alpha != 0.0);
    int64_t c, k;

    for (c = 0; c < N; ++c) {
        orow[c] = 0.0;
        if (mrow) mrow[c] = 0.0;
    }
    if (products) {
        /* Row i of op(A), widened to double (a copy, no arithmetic). */
        for (k = 0; k < K; ++k) arow[k] = a_at(j, i, k);
        if (!j->tb) {
            /* op(B) rows are contiguous: walk k in the outer loop so B is read
             * row by row.  Each orow[c] still receives its terms in ascending k. */
            for (k = 0; k < K; ++k) {
                const double a = arow[k];
                const float *brow = j->B + k * j->ldb;
                for (c = 0; c < N; ++c) orow[c] += a * (double)brow[c];
                if (mrow)
                    for (c = 0; c < N; ++c) mrow[c] += fabs(a) * fabs((double)brow[c]);
            }
        } else {
            for (c = 0; c < N; ++c) {
                double s = 0.0, m = 0.0;
                for (k = 0; k < K; ++k) {
                    const double b = b_at(j, k, c);
                    s += arow[k] * b;
                    m += fabs(arow[k]) * fabs(b);
                }
                orow[c] = s;
                if (mrow) mrow[c] = m;
            }
        }
    }
    for (c = 0; c < N; ++c) {
        double v = products ? j->alpha * orow[c] : 0.0;
        double m = (products && mrow) ? fabs(j->alpha) * mrow[c] : 0.0;
        if (j->beta != 0.0) {
            const double c0 = (double)j->C0[i * j->ldc + c];
            v += j->beta * c0;
            m += fabs(j->beta) * fabs(c0);
        }
        if (j->bias) {
            v += (double)j->bias[c];
            m += fabs((double)j->bias[c]);
        }
        if (j->row_bias) {
            v += (double)j->row_bias[i];
            m += fabs((double)j->row_bias[i]);
        }
        if (j->relu) v = (v > 0.0) ? v : 0.0;
        orow[c] = v;
        if (mrow) mrow[c] = m;
    }
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    double *arow = (double *)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
    int64_t r;
    if (!arow) {
        j->status = ORACLE_ENOMEM;
        return NULL;
    }
    for (r = j->first; r < j->last; ++r) {
        const int64_t i = j->rows ? j->rows[r] : r;
        one_row(j, i, j->out + r * j->N, j->mag ? j->mag + r * j->N : NULL, arow);
    }
    free(arow);
    j->status = ORACLE_OK;
    return NULL;
}

/*
 * Single GEMM.  Returns 0 on success.  `out` (and `mag`, if not NULL) receive
 * nrows x N doubles; with rows == NULL, nrows must equal M and row r of the
 * output is row r of C.  Otherwise row r of the output is row rows[r] of C.
 */
int oracle_gemm(int ta, int tb, int64_t M, int64_t N, int64_t K, float alpha,
                const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                const float *C0, int64_t ldc, const float *bias, const float *row_bias, int relu,
                const int64_t *rows, int64_t nrows, double *out, double *mag, int nthreads)
{
    job_t base;
    job_t *jobs;
    pthread_t *tids;
    int64_t r, per;
    int t, nt, rc = ORACLE_OK;

    if (M < 0 || N < 0 || K < 0 || nrows < 0 || (ta != 0 && ta != 1) || (tb != 0 && tb != 1))
        return ORACLE_EINVAL;
    if (!rows && nrows != M) return ORACLE_EINVAL;
    for (r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return ORACLE_EINVAL;
    if (nrows == 0 || N == 0) return ORACLE_OK;
    if (!out) return ORACLE_EINVAL;
    if (K > 0 && alpha != 0.0f && (!A || !B)) return ORACLE_EINVAL;
    if (beta != 0.0f && !C0) return ORACLE_EINVAL;

    memset(&base, 0, sizeof(base));
    base.ta = ta;
    base.tb = tb;
    base.M = M;
    base.N = N;
    base.K = K;
    base.alpha = (double)alpha;
    base.beta = (double)beta;
    base.A = A;
    base.lda = lda;
    base.B = B;
    base.ldb = ldb;
    base.C0 = C0;
    base.ldc = ldc;
    base.bias = bias;
    base.row_bias = row_bias;
    base.relu = relu ? 1 : 0;
    base.rows = rows;
    base.nrows = nrows;
    base.out = out;
    base.mag = mag;

    nt = nthreads < 1 ? 1 : nthreads;
    if ((int64_t)nt > nrows) nt = (int)nrows;
    jobs = (job_t *)calloc((size_t)nt, sizeof(job_t));
    tids = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return ORACLE_ENOMEM;
    }
    per = (nrows + nt - 1) / nt;
    for (t = 0; t < nt; ++t) {
        jobs[t] = base;
        jobs[t].first = (int64_t)t * per;
        jobs[t].last = jobs[t].first + per < nrows ? jobs[t].first + per : nrows;
        jobs[t].status = ORACLE_ENOMEM;
    }
    if (nt == 1) {
        worker(&jobs[0]);
    } else {
        for (t = 0; t < nt; ++t)
            if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0) {
                /* Run the slice on this thread instead. */
                tids[t] = 0;
                worker(&jobs[t]);
            }
        for (t = 0; t < nt; ++t)
            if (tids[t]) pthread_join(tids[t], NULL);
    }
    for (t = 0; t < nt; ++t)
        if (jobs[t].status != ORACLE_OK) rc = jobs[t].status;
    free(jobs);
    free(tids);
    return rc;
}

/*
 * Strided batch: problem b uses A + b*strideA, B + b*strideB, C0 + b*strideC and
 * writes its M x N result to out + b*M*N (and mag likewise).  The batched
 * operation is, by definition, the independent problems one after another.
 */
int oracle_gemm_strided_batched(int ta, int tb, int64_t M, int64_t N, int64_t K, float alpha,
                                const float *A, int64_t lda, int64_t strideA,
                                const float *B, int64_t ldb, int64_t strideB, float beta,
                                const float *C0, int64_t ldc, int64_t strideC, int64_t batch,
                                double *out, double *mag, int nthreads)
{
    int64_t b;
    if (batch < 0) return ORACLE_EINVAL;
    for (b = 0; b < batch; ++b) {
        const int rc = oracle_gemm(ta, tb, M, N, K, alpha, A ? A + b * strideA : NULL, lda,
                                   B ? B + b * strideB : NULL, ldb, beta,
                                   C0 ? C0 + b * strideC : NULL, ldc, NULL, NULL, 0, NULL, M,
                                   out + b * M * N, mag ? mag + b * M * N : NULL, nthreads);
        if (rc != ORACLE_OK) return rc;
    }
    return ORACLE_OK;
}

/*
 * spops_oracle.c -- plain fp64 CPU oracle for the CSR sparse-adapter operators.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the bench's
 * CPU-baseline leg load this library. The product (the CUDA library and its Python
 * binding) never calls it, shares no code with it and must fail loudly without its own
 * CUDA build. The oracle is slow on purpose: every result is the plain definition of the
 * operation, written out with fp64 arithmetic, one row at a time.
 *
 * Sources (spops README, "Sparse Operations (spops)"):
 *   - section "Usage": the CSR lists (values, row_offsets, col_idx, row_idx);
 *   - "Sparse Addition [dense = sparse + dense]": csr_add;
 *   - "Sparse Matrix Multiplication (SpMM) [dense = sparse x dense]": spmm;
 *   - "Sampled Dense-Dense Matrix Multiplication (SDDMM) [sparse = dense x dense]": sddmm,
 *     with BT the transpose of the right operand;
 *   - "Important Notes": row_offsets int32, other index lists int16.
 * torchsparsegradutils README, "Basic Sparse Matrix Multiplication": the gradient of a
 * sparse x dense product with respect to the sparse values is the sampled product, which
 * ties SDDMM to SpMM (tests check that adjoint identity on the oracle); the gradient with
 * respect to the dense operand is the transposed sparse matrix times the output gradient,
 * hence csr_transpose (spops README, "csr_transpose" in the operation list).
 * SparseAdam page (tensorplay.optim.sparse_adam.SparseAdam): Adam restricted to the
 * entries the sparse gradient materializes -- masked_adam.
 *
 * Readings where the pages leave a step open:
 *   - row_idx sorts rows by nnz in DESCENDING order; equal counts keep ascending row id;
 *   - SDDMM does not scale by any mask value (the call takes no values);
 *   - results are rounded once, round-to-nearest-even, to the operand dtype;
 *   - row bins are counted (rows with nnz >= t_long, rows with nnz >= 1), so they are
 *     defined for any row permutation;
 *   - the transpose is canonical CSR: row j of A^T lists column j of A by ascending row;
 *   - masked Adam uses the Adam update with bias-corrected moments,
 *     p -= lr * mhat / (sqrt(vhat) + eps), mhat = m / (1 - beta1^t), vhat = v / (1 - beta2^t),
 *     on the materialized entries only (the page lists the defaults and the masking, not the
 *     formula); maximize ascends.
 *
 * Parity pins: every function here is checked in the CPU test suite against brute force,
 * closed forms, library routines or the pages' worked structures. None is unpinned.
 *
 * Index arrays are int32 here; callers widen int16 lists before the call.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the parallel loops below use from now on (timing only; results do not depend on
 * it: each output row is computed by one thread in a fixed order). */
void oracle_set_threads(int32_t n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ row permutation */

static int cmp_i64(const void* a, const void* b) {
    int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

/* row_idx: the rows 0..m-1 ordered by nnz_i = ro[i+1]-ro[i], largest first, equal
 * counts by ascending row id. Sort key (INT32_MAX - nnz_i, i), ascending. */
int oracle_sort_rows(int32_t m, const int32_t* ro, int32_t* row_idx) {
    if (m <= 0) return 0;
    int64_t* key = (int64_t*)malloc(sizeof(int64_t) * (size_t)m);
    if (!key) return -1;
    for (int32_t i = 0; i < m; ++i) {
        int64_t nnz_i = (int64_t)ro[i + 1] - (int64_t)ro[i];
        key[i] = ((int64_t)(INT32_MAX - nnz_i) << 32) | (int64_t)i;
    }
    qsort(key, (size_t)m, sizeof(int64_t), cmp_i64);
    for (int32_t i = 0; i < m; ++i) row_idx[i] = (int32_t)(key[i] & 0xffffffffLL);
    free(key);
    return 0;
}

/* Row bins as prefix offsets along a row permutation sorted by sort_rows:
 * bins[0] = 0, bins[1] = #rows with nnz >= t_long, bins[2] = #rows with nnz >= 1,
 * bins[3] = m. Rows [bins[0], bins[1]) are long, [bins[1], bins[2]) short,
 * [bins[2], bins[3]) empty. */
int oracle_row_bins(int32_t m, const int32_t* ro, int32_t t_long, int32_t* bins) {
    int32_t nlong = 0, nonempty = 0;
    for (int32_t i = 0; i < m; ++i) {
        int32_t c = ro[i + 1] - ro[i];
        if (c >= t_long) ++nlong;
        if (c >= 1) ++nonempty;
    }
    bins[0] = 0;
    bins[1] = nlong;
    bins[2] = nonempty;
    bins[3] = m;
    return 0;
}

/* ------------------------------------------------------------------ operators */

/* SpMM: C[i, :] = sum over k in row i, in CSR order, of val[k] * B[col[k], :].
 * B is kdim x n row-major. With rows == NULL, C is m x n; otherwise C is nrows x n and
 * output row r holds sparse row rows[r]. Rows without entries give zeros. */
void oracle_spmm(int32_t m, int32_t kdim, int32_t n, const int32_t* ro, const int32_t* col,
                 const double* val, const double* B, double* C, const int32_t* rows,
                 int32_t nrows) {
    (void)kdim;
    int32_t count = rows ? nrows : m;
#pragma omp parallel for schedule(dynamic, 8)
    for (int32_t r = 0; r < count; ++r) {
        int32_t i = rows ? rows[r] : r;
        double* c = C + (int64_t)r * n;
        for (int32_t j = 0; j < n; ++j) c[j] = 0.0;
        for (int32_t k = ro[i]; k < ro[i + 1]; ++k) {
            const double a = val[k];
            const double* b = B + (int64_t)col[k] * n;
            for (int32_t j = 0; j < n; ++j) c[j] += a * b[j];
        }
    }
}

/* SDDMM: out[k] = sum_t A[i, t] * BT[col[k], t] for every entry k of row i.
 * A is m x kd, BT is n x kd, both row-major. With rows == NULL, out has nnz entries in
 * CSR order. Otherwise A holds only the selected rows (nrows x kd, row r <-> rows[r]) and
 * out holds their entries concatenated in the order of `rows`. */
void oracle_sddmm(int32_t m, int32_t n, int32_t kd, const int32_t* ro, const int32_t* col,
                  const double* A, const double* BT, double* out, const int32_t* rows,
                  int32_t nrows) {
    (void)n;
    int32_t count = rows ? nrows : m;
    int64_t* base = (int64_t*)malloc(sizeof(int64_t) * ((size_t)count + 1));
    if (!base) return;
    base[0] = 0;
    for (int32_t r = 0; r < count; ++r) {
        int32_t i = rows ? rows[r] : r;
        base[r + 1] = base[r] + (ro[i + 1] - ro[i]);
    }
#pragma omp parallel for schedule(dynamic, 8)
    for (int32_t r = 0; r < count; ++r) {
        int32_t i = rows ? rows[r] : r;
        const double* a = A + (int64_t)r * kd;
        for (int32_t k = ro[i]; k < ro[i + 1]; ++k) {
            const double* bt = BT + (int64_t)col[k] * kd;
            double s = 0.0;
            for (int32_t t = 0; t < kd; ++t) s += a[t] * bt[t];
            out[base[r] + (k - ro[i])] = s;
        }
    }
    free(base);
}

/* csr_add: C = B + A, with A the CSR matrix made dense (A[i, col[k]] = val[k]).
 * B and C are m x n row-major; with rows != NULL, B and C hold only the selected rows. */
void oracle_csr_add(int32_t m, int32_t n, const int32_t* ro, const int32_t* col,
                    const double* val, const double* B, double* C, const int32_t* rows,
                    int32_t nrows) {
    int32_t count = rows ? nrows : m;
#pragma omp parallel for schedule(static)
    for (int32_t r = 0; r < count; ++r) {
        int32_t i = rows ? rows[r] : r;
        const double* b = B + (int64_t)r * n;
        double* c = C + (int64_t)r * n;
        for (int32_t j = 0; j < n; ++j) c[j] = b[j];
        for (int32_t k = ro[i]; k < ro[i + 1]; ++k) c[col[k]] = b[col[k]] + val[k];
    }
}

/* ------------------------------------------------------------------ transpose */

/* A^T of an m x n CSR matrix, as an n x m CSR matrix: ro_t[j] counts the entries with
 * column < j; the entries of column j follow in ascending row order (the order in which a
 * walk over A's rows meets them). perm[p] is the entry of A placed at position p. */
void oracle_csr_transpose(int32_t m, int32_t n, const int32_t* ro, const int32_t* col, const double* val,
                          int32_t* ro_t, int32_t* row_t, double* val_t, int32_t* perm) {
    for (int32_t j = 0; j <= n; ++j) ro_t[j] = 0;
    for (int32_t i = 0; i < m; ++i)
        for (int32_t k = ro[i]; k < ro[i + 1]; ++k) ro_t[col[k] + 1] += 1;
    for (int32_t j = 0; j < n; ++j) ro_t[j + 1] += ro_t[j];
    int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    for (int32_t j = 0; j < n; ++j) next[j] = ro_t[j];
    for (int32_t i = 0; i < m; ++i) {
        for (int32_t k = ro[i]; k < ro[i + 1]; ++k) {
            const int32_t p = next[col[k]]++;
            row_t[p] = i;
            val_t[p] = val[k];
            perm[p] = k;
        }
    }
    free(next);
}

/* ------------------------------------------------------------------ masked Adam */

/* One Adam step (step number t >= 1) on the entries pos[g] of the parameter, g < count,
 * with gradient grad[g]; every other entry of param, exp_avg and exp_avg_sq is left as it
 * is. pos == NULL means pos[g] = g. */
void oracle_masked_adam(int64_t count, const int64_t* pos, const double* grad, double* param, double* exp_avg,
                        double* exp_avg_sq, int32_t t, double lr, double beta1, double beta2, double eps,
                        int32_t maximize) {
    const double bc1 = 1.0 - pow(beta1, (double)t), bc2 = 1.0 - pow(beta2, (double)t);
    for (int64_t g = 0; g < count; ++g) {
        const int64_t q = pos ? pos[g] : g;
        const double d = maximize ? -grad[g] : grad[g];
        exp_avg[q] = beta1 * exp_avg[q] + (1.0 - beta1) * d;
        exp_avg_sq[q] = beta2 * exp_avg_sq[q] + (1.0 - beta2) * d * d;
        const double mhat = exp_avg[q] / bc1, vhat = exp_avg_sq[q] / bc2;
        param[q] -= lr * mhat / (sqrt(vhat) + eps);
    }
}

/* ------------------------------------------------------------------ rounding */

/* Round x to the nearest value of a binary floating-point format with p significand bits
 * (hidden bit included), minimum normal exponent emin and maximum exponent emax; ties go
 * to the even significand; results beyond the largest finite value become infinities.
 * This is IEEE 754 roundTiesToEven written from the format's definition:
 * the spacing of representable numbers at |x| is 2^(max(e, emin) - p + 1) where
 * 2^e <= |x| < 2^(e+1). Dividing by that spacing is exact (a power of two), rint() rounds
 * to an integer with ties to even under the default rounding mode, and multiplying back
 * is exact. */
static double round_format(double x, int p, int emin, int emax) {
    if (x == 0.0 || isnan(x) || isinf(x)) return x;
    int e2;
    frexp(fabs(x), &e2); /* |x| = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;
    if (e < emin) e = emin;
    double q = ldexp(1.0, e - p + 1);
    double y = rint(x / q) * q;
    double maxf = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(y) > maxf) return copysign(INFINITY, x);
    return y;
}

/* fmt: 0 = fp32 (p 24, emin -126, emax 127), 1 = fp16 (p 11, -14, 15),
 *      2 = bf16 (p 8, -126, 127). */
double oracle_round(double x, int32_t fmt) {
    switch (fmt) {
        case 0: return round_format(x, 24, -126, 127);
        case 1: return round_format(x, 11, -14, 15);
        case 2: return round_format(x, 8, -126, 127);
        default: return NAN;
    }
}

void oracle_round_array(const double* x, double* y, int64_t count, int32_t fmt) {
    for (int64_t i = 0; i < count; ++i) y[i] = oracle_round(x[i], fmt);
}

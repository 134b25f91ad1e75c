/*
 * Oracle for the left-side, lower-triangular, non-transposed, non-unit-diagonal
 * triangular solve  L * X = alpha * B  (X overwrites B), and, in
 * oracle_trsm_general, for every other TRSM variant (side, triangle,
 * transpose / conjugate transpose, unit diagonal) from its BLAS definition.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call this file.  It shares
 * no code, header or helper with the CUDA library and must never be used as a
 * fallback for it.
 *
 * What it computes (plain definition, no blocking, no reordering):
 *   "Hierarchical Shared Memory-Aware Optimization for TRSM on GPU Platforms"
 *   (developinglight.com summary, "One framework, several paths" and the
 *   opening paragraph): the tested operation is the left-side
 *   lower-triangular TRSM on square matrices.  Its plain meaning is
 *   X = L^{-1} (alpha B), where L is the lower triangle of A including the
 *   diagonal (the strictly upper part of A is never read).
 *   "SOLVE_TRI CUDA kernel for small matrices" (llama.cpp PR 17457, the first
 *   posted kernel, "Forward substitution" loop): row i of X is the row's right
 *   hand side minus the dot product of row i of L with the rows of X already
 *   solved, divided by the diagonal entry, with no guard against a zero
 *   diagonal.  The oracle restates that recurrence as mathematics:
 *       x_i = ( alpha b_i - sum_{k<i} L_ik x_k ) / L_ii ,   i = 0 .. m-1,
 *   evaluated independently for every right-hand-side column.
 *
 * Precision: every value is promoted exactly to double (f32 / complex64
 * storage) and the whole recurrence runs in double; the result is rounded to
 * the storage type once, at the end.  Complex products are the textbook
 * (ac - bd) + (ad + bc)i; complex quotients use Smith's 1962 algorithm
 * (R. L. Smith, "Algorithm 116: Complex division", CACM 5(8), 1962).
 *
 * alpha = 0 follows BLAS: the selected columns of B become zero and A is not
 * read.  Built with -ffp-contract=off so no fused multiply-add changes the
 * rounding between the x86 and Arm hosts.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F64 = 1, OR_C64 = 2, OR_C128 = 3 };
enum { OR_COL_MAJOR = 0, OR_ROW_MAJOR = 1 };

typedef struct { double re, im; } ocplx;

static ocplx c_mul(ocplx a, ocplx b) {
    ocplx r;
    r.re = a.re * b.re - a.im * b.im;
    r.im = a.re * b.im + a.im * b.re;
    return r;
}

static ocplx c_sub(ocplx a, ocplx b) {
    ocplx r;
    r.re = a.re - b.re;
    r.im = a.im - b.im;
    return r;
}

/* Smith's algorithm: scale by the larger of |c|, |d| to avoid overflow. */
static ocplx c_div(ocplx a, ocplx b) {
    ocplx r;
    double c = b.re, d = b.im;
    double ac = c < 0 ? -c : c, ad = d < 0 ? -d : d;
    if (ac >= ad) {
        double q = d / c, den = c + d * q;
        r.re = (a.re + a.im * q) / den;
        r.im = (a.im - a.re * q) / den;
    } else {
        double q = c / d, den = c * q + d;
        r.re = (a.re * q + a.im) / den;
        r.im = (a.im * q - a.re) / den;
    }
    return r;
}

/* Offset of logical element (row, col) of one matrix. */
static int64_t off(int layout, int64_t ld, int64_t row, int64_t col) {
    return layout == OR_COL_MAJOR ? col * ld + row : row * ld + col;
}

static double ld_real(const void *p, int dtype, int64_t i) {
    return dtype == OR_F32 ? (double)((const float *)p)[i] : ((const double *)p)[i];
}

static ocplx ld_cplx(const void *p, int dtype, int64_t i) {
    ocplx r;
    if (dtype == OR_C64) {
        r.re = (double)((const float *)p)[2 * i];
        r.im = (double)((const float *)p)[2 * i + 1];
    } else {
        r.re = ((const double *)p)[2 * i];
        r.im = ((const double *)p)[2 * i + 1];
    }
    return r;
}

static void st_real(void *p, int dtype, int64_t i, double v) {
    if (dtype == OR_F32) ((float *)p)[i] = (float)v;
    else ((double *)p)[i] = v;
}

static void st_cplx(void *p, int dtype, int64_t i, ocplx v) {
    if (dtype == OR_C64) {
        ((float *)p)[2 * i] = (float)v.re;
        ((float *)p)[2 * i + 1] = (float)v.im;
    } else {
        ((double *)p)[2 * i] = v.re;
        ((double *)p)[2 * i + 1] = v.im;
    }
}

/*
 * One group of right-hand-side columns of one system.  s holds m * w values
 * (row i, column c at s[i*w + c]).  Row i first receives alpha * b_i; at step
 * k (ascending) every later row subtracts L_ik x_k, and at step i the row is
 * divided by L_ii.  Each x_i therefore sees exactly the operations of
 *   x_i = (alpha b_i - L_i0 x_0 - L_i1 x_1 - ... - L_i,i-1 x_{i-1}) / L_ii
 * in that order; traversing L by columns only changes which row is updated
 * first, never the order of the terms within one row.
 */
static void solve_real_group(int dtype, int layout, int64_t m, double alpha,
                             const void *A, int64_t lda, void *B, int64_t ldb,
                             const int64_t *js, int64_t w, double *s) {
    for (int64_t i = 0; i < m; ++i)
        for (int64_t c = 0; c < w; ++c)
            s[i * w + c] = alpha * ld_real(B, dtype, off(layout, ldb, i, js[c]));
    for (int64_t k = 0; k < m; ++k) {
        const double d = ld_real(A, dtype, off(layout, lda, k, k));
        double *xk = s + k * w;
        for (int64_t c = 0; c < w; ++c) xk[c] = xk[c] / d;
        for (int64_t i = k + 1; i < m; ++i) {
            const double l = ld_real(A, dtype, off(layout, lda, i, k));
            double *si = s + i * w;
            for (int64_t c = 0; c < w; ++c) si[c] -= l * xk[c];
        }
    }
    for (int64_t i = 0; i < m; ++i)
        for (int64_t c = 0; c < w; ++c)
            st_real(B, dtype, off(layout, ldb, i, js[c]), s[i * w + c]);
}

static void solve_cplx_group(int dtype, int layout, int64_t m, ocplx alpha,
                             const void *A, int64_t lda, void *B, int64_t ldb,
                             const int64_t *js, int64_t w, ocplx *s) {
    for (int64_t i = 0; i < m; ++i)
        for (int64_t c = 0; c < w; ++c)
            s[i * w + c] = c_mul(alpha, ld_cplx(B, dtype, off(layout, ldb, i, js[c])));
    for (int64_t k = 0; k < m; ++k) {
        const ocplx d = ld_cplx(A, dtype, off(layout, lda, k, k));
        ocplx *xk = s + k * w;
        for (int64_t c = 0; c < w; ++c) xk[c] = c_div(xk[c], d);
        for (int64_t i = k + 1; i < m; ++i) {
            const ocplx l = ld_cplx(A, dtype, off(layout, lda, i, k));
            ocplx *si = s + i * w;
            for (int64_t c = 0; c < w; ++c) si[c] = c_sub(si[c], c_mul(l, xk[c]));
        }
    }
    for (int64_t i = 0; i < m; ++i)
        for (int64_t c = 0; c < w; ++c)
            st_cplx(B, dtype, off(layout, ldb, i, js[c]), s[i * w + c]);
}

static int64_t elem_size(int dtype) {
    switch (dtype) {
    case OR_F32: return 4;
    case OR_F64: return 8;
    case OR_C64: return 8;
    default: return 16;
    }
}

/*
 * X = L^{-1}(alpha B) for `batch` systems, in place in B.
 *   dtype  0 f32, 1 f64, 2 complex64, 3 complex128 (interleaved re, im)
 *   layout 0 column-major, 1 row-major (per system)
 *   alpha  host pointer to two doubles (re, im); im ignored for real types
 *   cols   optional list of RHS column indices to solve (NULL = all n);
 *          columns not listed are left untouched
 *   nthreads  OpenMP threads (<= 0: runtime default)
 * Returns 0, or -k when argument k (1-based) is invalid.
 */
int oracle_trsm_llnn(int dtype, int layout, int64_t m, int64_t n, const double *alpha,
                     const void *A, int64_t lda, int64_t strideA,
                     void *B, int64_t ldb, int64_t strideB, int64_t batch,
                     const int64_t *cols, int64_t ncols, int nthreads) {
    if (dtype < 0 || dtype > 3) return -1;
    if (layout != OR_COL_MAJOR && layout != OR_ROW_MAJOR) return -2;
    if (m < 0) return -3;
    if (n < 0) return -4;
    if (!alpha) return -5;
    if (batch < 0) return -12;
    if (cols == NULL) ncols = n;
    if (ncols < 0) return -14;
    if (m == 0 || ncols == 0 || batch == 0) return 0;
    if (!B) return -9;
    const int cplx = dtype >= OR_C64;
    const int zero_alpha = alpha[0] == 0.0 && (!cplx || alpha[1] == 0.0);
    if (!zero_alpha && !A) return -6;
    const int64_t es = elem_size(dtype);
    /* work units: (system, group of up to GROUP consecutive listed columns) */
    enum { GROUP = 4 };
    const int64_t groups = (ncols + GROUP - 1) / GROUP;
    const int64_t units = batch * groups;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        void *s = malloc((size_t)m * GROUP * (cplx ? sizeof(ocplx) : sizeof(double)));
        int64_t js[GROUP];
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t u = 0; u < units; ++u) {
            const int64_t b = u / groups, g = u % groups;
            const int64_t c0 = g * GROUP;
            const int64_t w = ncols - c0 < GROUP ? ncols - c0 : GROUP;
            for (int64_t c = 0; c < w; ++c) js[c] = cols ? cols[c0 + c] : c0 + c;
            const char *Ab = (const char *)A + b * strideA * es;
            char *Bb = (char *)B + b * strideB * es;
            if (zero_alpha) {
                for (int64_t c = 0; c < w; ++c)
                    for (int64_t i = 0; i < m; ++i) {
                        if (cplx) { ocplx z = {0.0, 0.0}; st_cplx(Bb, dtype, off(layout, ldb, i, js[c]), z); }
                        else st_real(Bb, dtype, off(layout, ldb, i, js[c]), 0.0);
                    }
            } else if (cplx) {
                ocplx a = {alpha[0], alpha[1]};
                solve_cplx_group(dtype, layout, m, a, Ab, lda, Bb, ldb, js, w, (ocplx *)s);
            } else {
                solve_real_group(dtype, layout, m, alpha[0], Ab, lda, Bb, ldb, js, w, (double *)s);
            }
        }
        free(s);
    }
    (void)nthreads;
    return 0;
}

/*
 * Every TRSM variant, from its BLAS definition (the pages call the variants
 * beyond left/lower/no-transpose "other TRSM variants"; their meaning is the
 * standard xTRSM one):
 *   side 0 (left):   op(A) X = alpha B,  A is m x m
 *   side 1 (right):  X op(A) = alpha B,  A is n x n
 *   op(A) = A (trans 0), A^T (1) or A^H (2; A^T for real types); only the
 *   triangle `uplo` (0 lower, 1 upper) of A is read; diag 1 (unit) takes the
 *   diagonal as 1 without reading it.  Column-major, one system, serial.
 * The triangular matrix T = op(A) is read entry by entry through t_entry();
 * the substitution runs in the order T's shape dictates: for the left side
 * forward (T lower) or backward (T upper) over the rows of X, for the right
 * side forward (T upper) or backward (T lower) over its columns, each x
 * being (alpha b - the sum of the already solved terms, in the order they
 * were solved) / T_jj.  Double precision throughout, one rounding at the end.
 * Returns 0, or -k when argument k is invalid.
 */
static ocplx t_entry(int dtype, int uplo, int trans, int diag, const void *A, int64_t lda, int64_t i,
                     int64_t j) {
    ocplx v = {0.0, 0.0};
    if (i == j && diag == 1) {
        v.re = 1.0;
        return v;
    }
    /* T(i, j) = A(i, j), A(j, i) or conj(A(j, i)) */
    const int64_t r = trans ? j : i, c = trans ? i : j;
    if ((uplo == 0 && r < c) || (uplo == 1 && r > c)) return v; /* outside the referenced triangle */
    if (dtype >= OR_C64) {
        v = ld_cplx(A, dtype, c * lda + r);
        if (trans == 2) v.im = -v.im;
    } else {
        v.re = ld_real(A, dtype, c * lda + r);
    }
    return v;
}

int oracle_trsm_general(int dtype, int side, int uplo, int trans, int diag, int64_t m, int64_t n,
                        const double *alpha, const void *A, int64_t lda, void *B, int64_t ldb) {
    if (dtype < 0 || dtype > 3) return -1;
    if (side != 0 && side != 1) return -2;
    if (uplo != 0 && uplo != 1) return -3;
    if (trans < 0 || trans > 2) return -4;
    if (diag != 0 && diag != 1) return -5;
    if (m < 0) return -6;
    if (n < 0) return -7;
    if (!alpha) return -8;
    const int64_t k = side == 0 ? m : n;
    if (lda < (k > 1 ? k : 1)) return -10;
    if (ldb < (m > 1 ? m : 1)) return -12;
    if (m == 0 || n == 0) return 0;
    if (!B) return -11;
    const int cplx = dtype >= OR_C64;
    const int zero_alpha = alpha[0] == 0.0 && (!cplx || alpha[1] == 0.0);
    if (!zero_alpha && !A) return -9;
    const ocplx al = {alpha[0], cplx ? alpha[1] : 0.0};
    /* T lower when the referenced triangle is lower and not transposed, or upper and transposed */
    const int t_lower = (uplo == 0) != (trans != 0);
    ocplx *x = (ocplx *)malloc((size_t)k * sizeof(ocplx));
    const int64_t systems = side == 0 ? n : m; /* columns (left) or rows (right) of X */
    for (int64_t s = 0; s < systems; ++s) {
        /* the vector being solved: column s of B (left) or row s of B (right) */
        for (int64_t q = 0; q < k; ++q) {
            const int64_t o = side == 0 ? s * ldb + q : q * ldb + s;
            ocplx b = cplx ? ld_cplx(B, dtype, o) : (ocplx){ld_real(B, dtype, o), 0.0};
            x[q] = zero_alpha ? (ocplx){0.0, 0.0} : c_mul(al, b);
        }
        if (!zero_alpha) {
            /* left: T x = rhs (x a column); right: x T = rhs, i.e. T^T x = rhs */
            const int lower_system = side == 0 ? t_lower : !t_lower;
            for (int64_t step = 0; step < k; ++step) {
                const int64_t j = lower_system ? step : k - 1 - step;
                ocplx acc = x[j];
                for (int64_t st = 0; st < step; ++st) {
                    const int64_t q = lower_system ? st : k - 1 - st;
                    const ocplx tv = side == 0 ? t_entry(dtype, uplo, trans, diag, A, lda, j, q)
                                               : t_entry(dtype, uplo, trans, diag, A, lda, q, j);
                    acc = c_sub(acc, c_mul(tv, x[q]));
                }
                x[j] = c_div(acc, t_entry(dtype, uplo, trans, diag, A, lda, j, j));
            }
        }
        for (int64_t q = 0; q < k; ++q) {
            const int64_t o = side == 0 ? s * ldb + q : q * ldb + s;
            if (cplx) st_cplx(B, dtype, o, x[q]);
            else st_real(B, dtype, o, x[q].re);
        }
    }
    free(x);
    return 0;
}

/* Threads an OpenMP region would use by default (reported by the baseline). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

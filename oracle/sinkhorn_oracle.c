/*
 * Float64 CPU oracle for log-domain Sinkhorn with squared-Euclidean cost.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * It follows "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU"
 * (gist.science technical summary, read in its Korean, French and Chinese
 * versions), written out as plainly as possible:
 *   - Problem statement: entropic OT between weighted point clouds,
 *     cost C_ij = ||x_i - y_j||^2, solved by Sinkhorn iterations.
 *   - Method 1 (attention-form reformulation): the stabilised log-domain
 *     update f_i <- -eps LSE_j[(g_j - C_ij)/eps + log b_j], and Proposition 1,
 *     which rewrites it as a row LSE of S_X = (Q K^T + 1 (g_hat + delta)^T)/eps
 *     with Q = sqrt(2) X, K = sqrt(2) Y.
 *   - Method 3 (differentiation): transport-plan application
 *     (barycentric projection, gradient) as a weighted mean over the plan.
 * Readings of what the pages leave open:
 *   - the g-update is the symmetric one, g_j <- -eps LSE_i[(f_i - C_ij)/eps
 *     + log a_i] (the pages name gamma as the second log-weight bias);
 *   - one iteration = f-update from g, then g-update from the new f;
 *   - P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps);
 *   - g_hat_j = g_j - ||y_j||^2, delta_j = eps log b_j (the only choice under
 *     which Proposition 1 is an identity).
 *
 * Everything is float64 with libm exp/log, no fast-math, sums in index order.
 * OpenMP parallelises independent rows or columns only; every individual
 * reduction runs sequentially in index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int t) {
#ifdef _OPENMP
    if (t > 0) omp_set_num_threads(t);
#else
    (void)t;
#endif
}

/* ||x_i - y_j||^2 in the difference form, straight from the problem statement. */
static double sqdist(const float* x, const float* y, int d) {
    double s = 0.0;
    for (int k = 0; k < d; ++k) {
        double t = (double)x[k] - (double)y[k];
        s += t * t;
    }
    return s;
}

/* C (n x m, row-major, double) = squared Euclidean cost. */
void orc_cost(const float* X, int64_t n, const float* Y, int64_t m, int d, double* C) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < m; ++j)
            C[i * m + j] = sqdist(X + i * d, Y + j * d, d);
}

/* C (n x m, double) = cosine cost, written from its definition
 * C_ij = 2 - 2 cos(x_i, y_j) = 2 - 2 x_i.y_j / (|x_i| |y_j|)
 * (the pages' Discussion: the cosine cost is the squared-Euclidean cost of
 * the normalised points).  A zero row is taken as the zero vector after
 * normalisation, so its cost to a nonzero point is 1 and to a zero point 0:
 * C_ij = [x_i != 0] + [y_j != 0] - 2 x_i.y_j / (|x_i| |y_j|), the last term
 * 0 when either norm is 0. */
void orc_cost_cosine(const float* X, int64_t n, const float* Y, int64_t m, int d, double* C) {
    double* ny = (double*)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    for (int64_t j = 0; j < m; ++j) {
        double s = 0.0;
        for (int k = 0; k < d; ++k) s += (double)Y[j * d + k] * (double)Y[j * d + k];
        ny[j] = sqrt(s);
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int k = 0; k < d; ++k) s += (double)X[i * d + k] * (double)X[i * d + k];
        const double nx = sqrt(s);
        for (int64_t j = 0; j < m; ++j) {
            double dot = 0.0;
            for (int k = 0; k < d; ++k) dot += (double)X[i * d + k] * (double)Y[j * d + k];
            const double cosv = (nx > 0.0 && ny[j] > 0.0) ? dot / (nx * ny[j]) : 0.0;
            C[i * m + j] = (nx > 0.0 ? 1.0 : 0.0) + (ny[j] > 0.0 ? 1.0 : 0.0) - 2.0 * cosv;
        }
    }
    free(ny);
}

/* log sum_j exp(z_j), shifted by the maximum; sums in index order. */
static double lse(const double* z, int64_t len) {
    double M = -INFINITY;
    for (int64_t j = 0; j < len; ++j) if (z[j] > M) M = z[j];
    if (M == -INFINITY) return -INFINITY;
    double s = 0.0;
    for (int64_t j = 0; j < len; ++j) s += exp(z[j] - M);
    return M + log(s);
}

/* f-update (Method 1): f_i = -eps LSE_j[(g_j - C_ij)/eps + log b_j]. */
void orc_f_update(const double* C, int64_t n, int64_t m, const float* b, double eps,
                  const double* g, double* f) {
    double* lb = (double*)malloc(sizeof(double) * (size_t)m);
    for (int64_t j = 0; j < m; ++j) lb[j] = log((double)b[j]);
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)m);
#pragma omp for schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            for (int64_t j = 0; j < m; ++j)
                z[j] = (g[j] - C[i * m + j]) / eps + lb[j];
            f[i] = -eps * lse(z, m);
        }
        free(z);
    }
    free(lb);
}

/* g-update, the symmetric reading: g_j = -eps LSE_i[(f_i - C_ij)/eps + log a_i].
 * Each thread owns a block of columns and walks the rows of C in order, so
 * every column's maximum and sum run over i = 0..n-1 exactly as in lse(). */
void orc_g_update(const double* C, int64_t n, int64_t m, const float* a, double eps,
                  const double* f, double* g) {
    enum { JB = 64 };
    double* la = (double*)malloc(sizeof(double) * (size_t)n);
    for (int64_t i = 0; i < n; ++i) la[i] = log((double)a[i]);
    int64_t nblk = (m + JB - 1) / JB;
#pragma omp parallel for schedule(static)
    for (int64_t blk = 0; blk < nblk; ++blk) {
        int64_t j0 = blk * JB, j1 = j0 + JB < m ? j0 + JB : m;
        double M[JB], s[JB];
        for (int64_t j = j0; j < j1; ++j) { M[j - j0] = -INFINITY; s[j - j0] = 0.0; }
        for (int64_t i = 0; i < n; ++i)
            for (int64_t j = j0; j < j1; ++j) {
                double z = (f[i] - C[i * m + j]) / eps + la[i];
                if (z > M[j - j0]) M[j - j0] = z;
            }
        for (int64_t i = 0; i < n; ++i)
            for (int64_t j = j0; j < j1; ++j) {
                double z = (f[i] - C[i * m + j]) / eps + la[i];
                s[j - j0] += exp(z - M[j - j0]);
            }
        for (int64_t j = j0; j < j1; ++j)
            g[j] = -eps * (M[j - j0] + log(s[j - j0]));
    }
    free(la);
}

/* n_iter iterations, each an f-update from g followed by a g-update from the
 * new f.  f and g are in/out; g on entry seeds the first f-update. */
void orc_sinkhorn(const double* C, int64_t n, int64_t m, const float* a, const float* b,
                  double eps, int n_iter, double* f, double* g) {
    for (int t = 0; t < n_iter; ++t) {
        orc_f_update(C, n, m, b, eps, g, f);
        orc_g_update(C, n, m, a, eps, f, g);
    }
}

/* f-update evaluated point by point for selected rows, without a cost matrix:
 * the same formula as orc_f_update, for rows[0..nrows). */
void orc_f_update_rows(const float* X, const float* Y, int64_t m, int d, const float* b,
                       double eps, const double* g, const int64_t* rows, int64_t nrows,
                       double* out) {
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)m);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            const float* x = X + rows[r] * d;
            for (int64_t j = 0; j < m; ++j)
                z[j] = (g[j] - sqdist(x, Y + j * d, d)) / eps + log((double)b[j]);
            out[r] = -eps * lse(z, m);
        }
        free(z);
    }
}

/* Proposition 1 form of the f-update: with Q = sqrt(2) X, K = sqrt(2) Y,
 * g_hat_j = g_j - ||y_j||^2 and delta_j = eps log b_j,
 *     S_X[i,j] = (Q_i . K_j + g_hat_j + delta_j) / eps,
 *     f_i      = ||x_i||^2 - eps LSE_j S_X[i,j].
 * Q_i . K_j is formed as the plain sum over k of (sqrt2 x_ik)(sqrt2 y_jk). */
void orc_f_update_prop1(const float* X, int64_t n, const float* Y, int64_t m, int d,
                        const float* b, double eps, const double* g, double* f) {
    const double r2 = sqrt(2.0);
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)m);
#pragma omp for schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            const float* x = X + i * d;
            double xx = 0.0;
            for (int k = 0; k < d; ++k) xx += (double)x[k] * (double)x[k];
            for (int64_t j = 0; j < m; ++j) {
                const float* y = Y + j * d;
                double qk = 0.0, yy = 0.0;
                for (int k = 0; k < d; ++k) {
                    qk += (r2 * (double)x[k]) * (r2 * (double)y[k]);
                    yy += (double)y[k] * (double)y[k];
                }
                double ghat = g[j] - yy;
                double delta = eps * log((double)b[j]);
                z[j] = (qk + ghat + delta) / eps;
            }
            f[i] = xx - eps * lse(z, m);
        }
        free(z);
    }
}

/* Plan application (Method 3): out_i = sum_j P_ij V_j with
 * P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps); V is m x k. */
void orc_apply_plan(const double* C, int64_t n, int64_t m, const float* a, const float* b,
                    double eps, const double* f, const double* g, const float* V, int k,
                    double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double* o = out + i * k;
        for (int c = 0; c < k; ++c) o[c] = 0.0;
        for (int64_t j = 0; j < m; ++j) {
            double p = (double)a[i] * (double)b[j] * exp((f[i] + g[j] - C[i * m + j]) / eps);
            for (int c = 0; c < k; ++c) o[c] += p * (double)V[j * k + c];
        }
    }
}

/* The same plan application for selected rows, without a cost matrix. */
void orc_apply_plan_rows(const float* X, const float* a, const float* Y, const float* b,
                         int64_t m, int d, double eps, const double* f, const double* g,
                         const float* V, int k, const int64_t* rows, int64_t nrows,
                         double* out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        double* o = out + r * k;
        for (int c = 0; c < k; ++c) o[c] = 0.0;
        for (int64_t j = 0; j < m; ++j) {
            double cij = sqdist(X + i * d, Y + j * d, d);
            double p = (double)a[i] * (double)b[j] * exp((f[i] + g[j] - cij) / eps);
            for (int c = 0; c < k; ++c) o[c] += p * (double)V[j * k + c];
        }
    }
}

/* Row sums P 1 (n) and column sums P^T 1 (m) of the plan. */
void orc_marginals(const double* C, int64_t n, int64_t m, const float* a, const float* b,
                   double eps, const double* f, const double* g, double* row, double* col) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int64_t j = 0; j < m; ++j)
            s += (double)a[i] * (double)b[j] * exp((f[i] + g[j] - C[i * m + j]) / eps);
        row[i] = s;
    }
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < m; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < n; ++i)
            s += (double)a[i] * (double)b[j] * exp((f[i] + g[j] - C[i * m + j]) / eps);
        col[j] = s;
    }
}

/* Transport cost <P, C>. */
double orc_transport_cost(const double* C, int64_t n, int64_t m, const float* a,
                          const float* b, double eps, const double* f, const double* g) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < m; ++j)
            s += (double)a[i] * (double)b[j] * exp((f[i] + g[j] - C[i * m + j]) / eps) *
                 C[i * m + j];
    return s;
}

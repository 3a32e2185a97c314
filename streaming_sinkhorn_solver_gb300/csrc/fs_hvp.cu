// Streaming Hessian-vector product of the converged entropic OT value with
// respect to X.
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 3 and
// the Discussion name a streaming Hessian-vector product built from
// transport-vector and transport-matrix products in O((n + m) d) memory but
// give no formula.  The one used here is derived from the fixed point:
//
//   F(X) = <a, f*> + <b, g*>,   grad_i = 2 (a_i x_i - (P Y)_i)
//   along X + t V:  d/dt P_ij = P_ij (fdot_i + gdot_j - Cdot_ij) / eps,
//                   Cdot_ij = 2 (x_i - y_j) . v_i = -2 t_ij,  t_ij = v_i . (y_j - x_i)
//   P 1 = a and P^T 1 = b differentiated:
//      a_i fdot_i + (P gdot)_i   = r_i = sum_j P_ij Cdot_ij = -2 sum_j P_ij t_ij
//      (P^T fdot)_j + b_j gdot_j = c_j = sum_i P_ij Cdot_ij = 2 (P^T w)_j - 2 y_j.(P^T V)_j
//   (w_i = x_i . v_i).  Eliminating fdot = (r - P gdot) / a leaves
//      S gdot = c - P^T (r / a),   S = diag(b) - P^T diag(1/a) P,
//   symmetric positive semi-definite with null space 1 (the gauge), solved by
//   conjugate gradients in the complement of 1.  Then
//   (H V)_i = 2 a_i v_i - (2/eps) [fdot_i (P Y)_i + (P (gdot . Y))_i + 2 T_i],
//   T_i = sum_j P_ij t_ij y_j.
// Every product with P or P^T is one streamed plan application of this
// library; T and sum_j P_ij t_ij come from one tangent application (the plan
// entries weighted by t_ij, a second dot-product tile U K^T beside the score
// tile on the tensor path, d more FMAs per pair on the FMA path).  Nothing
// of size n x m or n d^2 is stored: the scratch is O((n + m) d).
#include "fs_host.cuh"

#include <algorithm>
#include <cmath>

namespace fs {

namespace {

constexpr int kT = 256;

unsigned blocks_for(int64_t len) { return (unsigned)((len + kT - 1) / kT); }

// out_i = scale * sum_k A_ik B_ik
__global__ void k_rowdot(const float* __restrict__ A, const float* __restrict__ B, int64_t rows,
                         int d, float scale, float* __restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i >= rows) return;
    double s = 0.0;
    for (int k = 0; k < d; ++k) s += (double)A[i * d + k] * (double)B[i * d + k];
    out[i] = (float)(scale * s);
}

// r_i = -2 sum_j P_ij t_ij;  q_i = r_i / a_i
__global__ void k_hvp_r(const float* __restrict__ a, const float* __restrict__ pt, int64_t n,
                        float* __restrict__ r, float* __restrict__ q) {
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i >= n) return;
    const float ri = -2.f * pt[i];
    r[i] = ri;
    q[i] = ri / a[i];
}

// U_i = (w_i, v_i1, ..., v_id)
__global__ void k_pack_u(const float* __restrict__ w, const float* __restrict__ V, int64_t n,
                         int d, float* __restrict__ U) {
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i >= n) return;
    U[i * (d + 1)] = w[i];
    for (int k = 0; k < d; ++k) U[i * (d + 1) + 1 + k] = V[i * d + k];
}

// rhs_j = 2 PtU_j0 - 2 sum_k y_jk PtU_j(1+k) - t_j
__global__ void k_hvp_rhs(const float* __restrict__ PtU, const float* __restrict__ Y,
                          const float* __restrict__ t, int64_t m, int d, float* __restrict__ rhs) {
    const int64_t j = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (j >= m) return;
    double s = 0.0;
    for (int k = 0; k < d; ++k) s += (double)Y[j * d + k] * (double)PtU[j * (d + 1) + 1 + k];
    rhs[j] = (float)(2.0 * (double)PtU[j * (d + 1)] - 2.0 * s - (double)t[j]);
}

__global__ void k_add_scalar(float* __restrict__ v, int64_t len, float s) {
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i < len) v[i] += s;
}

// out_i = x_i / a_i
__global__ void k_div(const float* __restrict__ x, const float* __restrict__ a, int64_t len,
                      float* __restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i < len) out[i] = x[i] / a[i];
}

// Sp_j = b_j p_j - t_j
__global__ void k_sp(const float* __restrict__ b, const float* __restrict__ p,
                     const float* __restrict__ t, int64_t len, float* __restrict__ Sp) {
    const int64_t j = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (j < len) Sp[j] = b[j] * p[j] - t[j];
}

// x += alpha p;  res -= alpha Sp
__global__ void k_cg_update(float* __restrict__ x, float* __restrict__ res,
                            const float* __restrict__ p, const float* __restrict__ Sp, int64_t len,
                            float alpha) {
    const int64_t j = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (j >= len) return;
    x[j] += alpha * p[j];
    res[j] -= alpha * Sp[j];
}

// p = res + beta p
__global__ void k_cg_dir(float* __restrict__ p, const float* __restrict__ res, int64_t len,
                         float beta) {
    const int64_t j = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (j < len) p[j] = res[j] + beta * p[j];
}

// fdot_i = (r_i - Pg_i) / a_i
__global__ void k_fdot(const float* __restrict__ r, const float* __restrict__ pg,
                       const float* __restrict__ a, int64_t n, float* __restrict__ fdot) {
    const int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (i < n) fdot[i] = (r[i] - pg[i]) / a[i];
}

// Z_j = gdot_j y_j, one thread per element
__global__ void k_gy(const float* __restrict__ Y, const float* __restrict__ gdot, int64_t m, int d,
                     float* __restrict__ Z) {
    const int64_t e = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (e >= m * d) return;
    Z[e] = gdot[e / d] * Y[e];
}

// out_i = 2 a_i v_i - (2/eps) [fdot_i PY_i + PZ_i + 2 T_i], one thread per element
__global__ void k_hvp_final(const float* __restrict__ a, const float* __restrict__ V,
                            const float* __restrict__ fdot, const float* __restrict__ PY,
                            const float* __restrict__ PZ, const float* __restrict__ T, int64_t n,
                            int d, float two_over_eps, float* __restrict__ out) {
    const int64_t e = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (e >= n * d) return;
    const int64_t i = e / d;
    const double bracket = (double)fdot[i] * PY[e] + (double)PZ[e] + 2.0 * (double)T[e];
    out[e] = (float)(2.0 * (double)a[i] * V[e] - (double)two_over_eps * bracket);
}

struct Hvp {
    const float *X, *a, *Y, *b, *f, *g;
    int64_t n, m;
    int32_t d;
    float eps;
    const fs_options* opt;
    cudaStream_t s;
};

fs_status apply_p(const Hvp& h, const float* V, int32_t k, float* out) {
    return fs_apply_plan(h.X, h.a, h.n, h.Y, h.b, h.m, h.d, h.eps, h.f, h.g, V, k, out, h.opt, h.s);
}

fs_status apply_pt(const Hvp& h, const float* U, int32_t k, float* out) {
    return fs_apply_plan_t(h.X, h.a, h.n, h.Y, h.b, h.m, h.d, h.eps, h.f, h.g, U, k, out, h.opt,
                           h.s);
}

// one double, reduced on the GPU, read back (synchronises)
fs_status dot_host(const float* x, const float* y, int64_t len, double* partial, double* dres,
                   cudaStream_t s, double* out) {
    FS_CUDA(launch_dot_double(x, y, len, partial, dres, 0, s));
    FS_CUDA(cudaMemcpyAsync(out, dres, sizeof(double), cudaMemcpyDeviceToHost, s));
    FS_CUDA(cudaStreamSynchronize(s));
    return FS_OK;
}

fs_status hvp_entry(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                    int64_t m, int32_t d, float eps, const float* f, const float* g,
                    const float* V, float* out, int32_t cg_max_iter, float cg_tol,
                    const fs_options* opt, void* stream) {
    if (!X || !a || !Y || !b || !f || !g || !V || !out)
        return fail(FS_ERR_INVALID_ARG, "null pointer");
    if (n < 1 || m < 1) return fail(FS_ERR_INVALID_ARG, "n=%lld m=%lld", (long long)n, (long long)m);
    if (d < 1 || d > kMaxDim)
        return fail(FS_ERR_INVALID_ARG, "d=%d out of range [1, %d]", d, kMaxDim);
    if (!(eps > 0.f) || !std::isfinite(eps)) return fail(FS_ERR_INVALID_ARG, "eps must be positive");
    if (cg_max_iter < 0 || !(cg_tol >= 0.f)) return fail(FS_ERR_INVALID_ARG, "cg_max_iter/cg_tol");
    if (opt && opt->cost != FS_COST_SQEUCLIDEAN)
        return fail(FS_ERR_UNSUPPORTED, "fs_hvp_x is defined for the squared-Euclidean cost");
    const int max_iter = cg_max_iter > 0 ? cg_max_iter : 200;
    const double tol = cg_tol > 0.f ? (double)cg_tol : 1e-6;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Scratch sc(s);
    Hvp h{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, n, m, d, eps, opt, s};
    const float* V_d;
    FS_CUDA(sc.device_view(X, (size_t)n * d, &h.X));
    FS_CUDA(sc.device_view(a, (size_t)n, &h.a));
    FS_CUDA(sc.device_view(Y, (size_t)m * d, &h.Y));
    FS_CUDA(sc.device_view(b, (size_t)m, &h.b));
    FS_CUDA(sc.device_view(f, (size_t)n, &h.f));
    FS_CUDA(sc.device_view(g, (size_t)m, &h.g));
    FS_CUDA(sc.device_view(V, (size_t)n * d, &V_d));
    const bool out_dev = is_device_ptr(out);
    float* out_d = out;
    if (!out_dev) FS_CUDA(sc.get(&out_d, (size_t)n * d));

    float *PY, *T, *pt, *w, *r, *q, *U, *PtU, *t, *rhs, *x, *res, *p, *Sp, *tn, *tn2, *fdot, *Z,
        *PZ;
    double *partial, *dres;
    FS_CUDA(sc.get(&PY, (size_t)n * d));
    FS_CUDA(sc.get(&T, (size_t)n * d));
    FS_CUDA(sc.get(&pt, (size_t)n));
    FS_CUDA(sc.get(&w, (size_t)n));
    FS_CUDA(sc.get(&r, (size_t)n));
    FS_CUDA(sc.get(&q, (size_t)n));
    FS_CUDA(sc.get(&U, (size_t)n * (d + 1)));
    FS_CUDA(sc.get(&PtU, (size_t)m * (d + 1)));
    FS_CUDA(sc.get(&t, (size_t)m));
    FS_CUDA(sc.get(&rhs, (size_t)m));
    FS_CUDA(sc.get(&x, (size_t)m));
    FS_CUDA(sc.get(&res, (size_t)m));
    FS_CUDA(sc.get(&p, (size_t)m));
    FS_CUDA(sc.get(&Sp, (size_t)m));
    FS_CUDA(sc.get(&tn, (size_t)n));
    FS_CUDA(sc.get(&tn2, (size_t)n));
    FS_CUDA(sc.get(&fdot, (size_t)n));
    FS_CUDA(sc.get(&Z, (size_t)m * d));
    FS_CUDA(sc.get(&PZ, (size_t)n * d));
    FS_CUDA(sc.get(&partial, kRedPartials));
    FS_CUDA(sc.get(&dres, 1));
    float* ones = nullptr;
    FS_CUDA(sc.get(&ones, (size_t)m));

    // P Y, the tangent terms (T, sum_j P_ij t_ij), r and the right-hand side
    FS_TRY(apply_p(h, h.Y, d, PY));
    FS_TRY(apply_tangent(h.X, h.a, n, h.Y, h.b, m, d, eps, h.f, h.g, V_d, h.Y, d, T, pt, opt, s));
    k_hvp_r<<<blocks_for(n), kT, 0, s>>>(h.a, pt, n, r, q);
    k_rowdot<<<blocks_for(n), kT, 0, s>>>(h.X, V_d, n, d, 1.f, w);
    k_pack_u<<<blocks_for(n), kT, 0, s>>>(w, V_d, n, d, U);
    count_launch(3);
    FS_CUDA(cudaGetLastError());
    FS_TRY(apply_pt(h, U, d + 1, PtU));
    FS_TRY(apply_pt(h, q, 1, t));
    k_hvp_rhs<<<blocks_for(m), kT, 0, s>>>(PtU, h.Y, t, m, d, rhs);
    count_launch();
    FS_CUDA(cudaMemsetAsync(ones, 0, sizeof(float) * (size_t)m, s));
    k_add_scalar<<<blocks_for(m), kT, 0, s>>>(ones, m, 1.f);
    count_launch();
    FS_CUDA(cudaGetLastError());

    // the gauge direction 1 is the null space of S: keep the iteration in its complement
    auto project = [&](float* v) -> fs_status {
        double sum = 0.0;
        FS_TRY(dot_host(v, ones, m, partial, dres, s, &sum));
        k_add_scalar<<<blocks_for(m), kT, 0, s>>>(v, m, (float)(-sum / (double)m));
        count_launch();
        FS_CUDA(cudaGetLastError());
        return FS_OK;
    };
    FS_TRY(project(rhs));

    // conjugate gradients on S gdot = rhs from gdot = 0
    double bn2 = 0.0;
    FS_TRY(dot_host(rhs, rhs, m, partial, dres, s, &bn2));
    FS_CUDA(cudaMemsetAsync(x, 0, sizeof(float) * (size_t)m, s));
    FS_CUDA(cudaMemcpyAsync(res, rhs, sizeof(float) * (size_t)m, cudaMemcpyDeviceToDevice, s));
    FS_CUDA(cudaMemcpyAsync(p, rhs, sizeof(float) * (size_t)m, cudaMemcpyDeviceToDevice, s));
    double rr = bn2;
    for (int it = 0; it < max_iter && rr > tol * tol * bn2 && bn2 > 0.0; ++it) {
        FS_TRY(apply_p(h, p, 1, tn));
        k_div<<<blocks_for(n), kT, 0, s>>>(tn, h.a, n, tn2);
        count_launch();
        FS_TRY(apply_pt(h, tn2, 1, t));
        k_sp<<<blocks_for(m), kT, 0, s>>>(h.b, p, t, m, Sp);
        count_launch();
        FS_CUDA(cudaGetLastError());
        FS_TRY(project(Sp));
        double pSp = 0.0;
        FS_TRY(dot_host(p, Sp, m, partial, dres, s, &pSp));
        if (!(pSp > 0.0)) break;   // only the null direction is left
        const double alpha = rr / pSp;
        k_cg_update<<<blocks_for(m), kT, 0, s>>>(x, res, p, Sp, m, (float)alpha);
        count_launch();
        double rr_new = 0.0;
        FS_TRY(dot_host(res, res, m, partial, dres, s, &rr_new));
        k_cg_dir<<<blocks_for(m), kT, 0, s>>>(p, res, m, (float)(rr_new / rr));
        count_launch();
        FS_CUDA(cudaGetLastError());
        rr = rr_new;
    }

    // fdot, then the Hessian-vector product
    FS_TRY(apply_p(h, x, 1, tn));
    k_fdot<<<blocks_for(n), kT, 0, s>>>(r, tn, h.a, n, fdot);
    k_gy<<<blocks_for(m * (int64_t)d), kT, 0, s>>>(h.Y, x, m, d, Z);
    count_launch(2);
    FS_CUDA(cudaGetLastError());
    FS_TRY(apply_p(h, Z, d, PZ));
    k_hvp_final<<<blocks_for(n * (int64_t)d), kT, 0, s>>>(h.a, V_d, fdot, PY, PZ, T, n, d,
                                                          (float)(2.0 / (double)eps), out_d);
    count_launch();
    FS_CUDA(cudaGetLastError());
    if (!out_dev)
        FS_CUDA(cudaMemcpyAsync(out, out_d, sizeof(float) * (size_t)n * d, cudaMemcpyDeviceToHost, s));
    FS_CUDA(cudaStreamSynchronize(s));
    return FS_OK;
}

}  // namespace

// Device bytes of fs_hvp_x with device inputs: its stream-ordered scratch
// (the vectors allocated above) plus the largest library workspace its plan
// applications grow to (P with k = d, P^T with k = d + 1, the tangent).
int64_t hvp_workspace_bytes(int64_t n, int64_t m, int32_t d, const fs_options* opt) {
    const int64_t floats = n * (4 * (int64_t)d + 8) + m * (2 * (int64_t)d + 8);
    const int64_t own = 4 * floats + 8 * (kRedPartials + 1);
    int64_t ws = workspace_bytes_any(n, m, d, d, opt, false);
    ws = std::max(ws, workspace_bytes_any(m, n, d, d + 1, opt, false));
    ws = std::max(ws, workspace_bytes_any(n, m, d, d, opt, true));
    return ws < 0 ? -1 : own + ws;
}

}  // namespace fs

extern "C" int64_t fs_hvp_workspace_bytes(int64_t n, int64_t m, int32_t d, const fs_options* opt) {
    if (n < 1 || m < 1 || d < 1 || d > fs::kMaxDim) return -1;
    if (opt && opt->cost != FS_COST_SQEUCLIDEAN) return -1;
    return fs::hvp_workspace_bytes(n, m, d, opt);
}

extern "C" fs_status fs_hvp_x(const float* X, const float* a, int64_t n, const float* Y,
                              const float* b, int64_t m, int32_t d, float eps, const float* f,
                              const float* g, const float* V, float* out, int32_t cg_max_iter,
                              float cg_tol, const fs_options* opt, void* stream) {
    try {
        return fs::hvp_entry(X, a, n, Y, b, m, d, eps, f, g, V, out, cg_max_iter, cg_tol, opt,
                             stream);
    } catch (...) {
        return fs::fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

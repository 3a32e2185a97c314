// The cosine cost (FS_COST_COSINE).
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Discussion:
// the cosine cost C_ij = 2 - 2 cos(x_i, y_j) is the squared-Euclidean cost of
// the normalised points x^_i = x_i / |x_i|, y^_j = y_j / |y_j|, so the whole
// squared-Euclidean path runs unchanged on normalised copies of the clouds.
// Only the gradient with respect to the caller's x_i needs more: the chain
// rule through the normalisation, (I - x^ x^T) / |x| applied to the gradient
// at x^.  A zero row stays the zero vector (cost 1 to any unit point) and
// gets a zero gradient.
#include "fs_host.cuh"

namespace fs {

namespace {

constexpr int kCosWarps = 8;   // rows per 256-thread block, one warp each

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// out_i = p_i / |p_i| (0 for a zero row); norms_i = |p_i| (when not null)
__global__ void __launch_bounds__(32 * kCosWarps) k_normalize_rows(const float* __restrict__ P,
                                                                   int64_t rows, int d,
                                                                   float* __restrict__ out,
                                                                   float* __restrict__ norms) {
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kCosWarps + (threadIdx.x >> 5);
    if (r >= rows) return;
    const float* p = P + r * d;
    double s = 0.0;
    for (int k = lane; k < d; k += 32) s += (double)p[k] * (double)p[k];
    s = warp_sum(s);
    const double nrm = sqrt(s);
    const float inv = nrm > 0.0 ? (float)(1.0 / nrm) : 0.f;
    for (int k = lane; k < d; k += 32) out[r * d + k] = p[k] * inv;
    if (norms != nullptr && lane == 0) norms[r] = (float)nrm;
}

// G_i <- (G_i - (x^_i . G_i) x^_i) / |x_i|   (0 for a zero row)
__global__ void __launch_bounds__(32 * kCosWarps) k_project_grad(float* __restrict__ G,
                                                                 const float* __restrict__ Xn,
                                                                 const float* __restrict__ norms,
                                                                 int64_t rows, int d) {
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kCosWarps + (threadIdx.x >> 5);
    if (r >= rows) return;
    float* g = G + r * d;
    const float* x = Xn + r * d;
    double dot = 0.0;
    for (int k = lane; k < d; k += 32) dot += (double)x[k] * (double)g[k];
    dot = warp_sum(dot);
    const float nrm = norms[r];
    const float inv = nrm > 0.f ? 1.f / nrm : 0.f;
    const float dt = (float)dot;
    for (int k = lane; k < d; k += 32) g[k] = (g[k] - dt * x[k]) * inv;
}

unsigned cos_grid(int64_t rows) { return (unsigned)((rows + kCosWarps - 1) / kCosWarps); }

}  // namespace

void layout_cos(Layout& L, CosBufs& cb, const Problem& P) {
    if (P.cost != FS_COST_COSINE) return;
    cb.xn = L.take(sizeof(float) * (size_t)P.n * P.d);
    cb.yn = L.take(sizeof(float) * (size_t)P.m * P.d);
    cb.nx = L.take(sizeof(float) * (size_t)P.n);
    cb.used = true;
}

int64_t cos_workspace_bytes(int64_t n, int64_t m, int32_t d, const fs_options* opt) {
    if (!opt || opt->cost != FS_COST_COSINE) return 0;
    Layout L;
    L.take(sizeof(float) * (size_t)n * d);
    L.take(sizeof(float) * (size_t)m * d);
    L.take(sizeof(float) * (size_t)n);
    return (int64_t)L.off;
}

fs_status prepare_cos(Call& c, Problem& P, const CosBufs& cb, bool v_is_points) {
    if (!cb.used) return FS_OK;
    float* xn = c.at<float>(cb.xn);
    float* yn = c.at<float>(cb.yn);
    float* nx = c.at<float>(cb.nx);
    k_normalize_rows<<<cos_grid(P.n), 32 * kCosWarps, 0, c.stream>>>(P.X.dev, P.n, P.d, xn, nx);
    count_launch();
    FS_CUDA(cudaGetLastError());
    k_normalize_rows<<<cos_grid(P.m), 32 * kCosWarps, 0, c.stream>>>(P.Y.dev, P.m, P.d, yn,
                                                                     nullptr);
    count_launch();
    FS_CUDA(cudaGetLastError());
    // the barycentric map and the gradient use the points themselves as values
    if (v_is_points && P.V.alias == &P.Y) P.V.dev = yn;
    P.X.dev = xn;
    P.Y.dev = yn;
    return FS_OK;
}

fs_status finish_grad_cos(Call& c, Problem& P, const CosBufs& cb) {
    if (!cb.used) return FS_OK;
    k_project_grad<<<cos_grid(P.n), 32 * kCosWarps, 0, c.stream>>>(
        P.out.dev, c.at<float>(cb.xn), c.at<float>(cb.nx), P.n, P.d);
    count_launch();
    FS_CUDA(cudaGetLastError());
    return FS_OK;
}

}  // namespace fs

// Scalar reports on a solved problem: the dual value and the two marginal
// residuals of the plan.
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 1: the
// dual objective <a, f> + <b, g> (whose gradient Method 3 streams) and the
// marginal constraints P 1 = a, P^T 1 = b that the alternating updates
// enforce (the row sums equal a just after an f-update, the column sums b
// just after a g-update).  Both reductions run on the GPU in double, in a
// fixed order (one partial per block over a fixed index range, then the
// partials in block order), so the results are bitwise reproducible.
#include "fs_host.cuh"

#include <algorithm>
#include <vector>

namespace fs {

namespace {

constexpr int kRedThreads = 256;
constexpr int kRedMaxBlocks = kRedPartials;

// MODE 0: sum x_i y_i; MODE 1: sum |x_i - y_i|
template <int MODE>
__global__ void __launch_bounds__(kRedThreads) k_reduce(const float* __restrict__ x,
                                                        const float* __restrict__ y, int64_t len,
                                                        int64_t chunk, double* __restrict__ partial) {
    __shared__ double sh[kRedThreads];
    const int64_t start = (int64_t)blockIdx.x * chunk;
    const int64_t end = min(len, start + chunk);
    double acc = 0.0;
    for (int64_t i = start + threadIdx.x; i < end; i += kRedThreads) {
        const double xi = x[i], yi = y[i];
        acc += MODE == 0 ? xi * yi : fabs(xi - yi);
    }
    sh[threadIdx.x] = acc;
    __syncthreads();
#pragma unroll
    for (int w = kRedThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) partial[blockIdx.x] = sh[0];
}

// out[slot] (+)= sum of the partials in block order
__global__ void k_reduce_final(const double* __restrict__ partial, int nblk, double* out, int add) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    double s = 0.0;
    for (int i = 0; i < nblk; ++i) s += partial[i];
    *out = add ? *out + s : s;
}

__global__ void k_fill(float* __restrict__ v, int64_t len, float x) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < len) v[i] = x;
}

// Fixed block count and index range per block for a reduction of `len` terms.
int red_blocks(int64_t len, int64_t* chunk) {
    const int64_t nb = std::min<int64_t>(kRedMaxBlocks, (len + 4 * kRedThreads - 1) / (4 * kRedThreads));
    *chunk = (len + nb - 1) / nb;
    return (int)((len + *chunk - 1) / *chunk);
}

template <int MODE>
cudaError_t reduce_into(const float* x, const float* y, int64_t len, double* partial, double* out,
                        int add, cudaStream_t s) {
    int64_t chunk;
    const int nb = red_blocks(len, &chunk);
    k_reduce<MODE><<<nb, kRedThreads, 0, s>>>(x, y, len, chunk, partial);
    count_launch();
    k_reduce_final<<<1, 32, 0, s>>>(partial, nb, out, add);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dot_double(const float* x, const float* y, int64_t len, double* partial,
                              double* out, int add, cudaStream_t s) {
    return reduce_into<0>(x, y, len, partial, out, add, s);
}

cudaError_t launch_l1_double(const float* x, const float* y, int64_t len, double* partial,
                             double* out, int add, cudaStream_t s) {
    return reduce_into<1>(x, y, len, partial, out, add, s);
}

namespace {

fs_status dual_entry(const float* a, int64_t n, const float* b, int64_t m, const float* f,
                     const float* g, double* out, void* stream) {
    if (!a || !b || !f || !g || !out) return fail(FS_ERR_INVALID_ARG, "null pointer");
    if (n < 1 || m < 1) return fail(FS_ERR_INVALID_ARG, "n=%lld m=%lld", (long long)n, (long long)m);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Scratch sc(s);
    const float *ad, *bd, *fd, *gd;
    FS_CUDA(sc.device_view(a, (size_t)n, &ad));
    FS_CUDA(sc.device_view(b, (size_t)m, &bd));
    FS_CUDA(sc.device_view(f, (size_t)n, &fd));
    FS_CUDA(sc.device_view(g, (size_t)m, &gd));
    double *partial, *res;
    FS_CUDA(sc.get(&partial, kRedMaxBlocks));
    FS_CUDA(sc.get(&res, 1));
    FS_CUDA(reduce_into<0>(ad, fd, n, partial, res, 0, s));
    FS_CUDA(reduce_into<0>(bd, gd, m, partial, res, 1, s));
    FS_CUDA(cudaMemcpyAsync(out, res, sizeof(double), cudaMemcpyDeviceToHost, s));
    FS_CUDA(cudaStreamSynchronize(s));
    return FS_OK;
}

fs_status marginal_entry(const float* X, const float* a, int64_t n, const float* Y,
                         const float* b, int64_t m, int32_t d, float eps, const float* f,
                         const float* g, double* out, const fs_options* opt, void* stream) {
    if (!out) return fail(FS_ERR_INVALID_ARG, "null out");
    if (!a || !b) return fail(FS_ERR_INVALID_ARG, "null a or b");
    if (n < 1 || m < 1) return fail(FS_ERR_INVALID_ARG, "n=%lld m=%lld", (long long)n, (long long)m);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Scratch sc(s);
    float *ones, *rows, *cols;
    double *partial, *res;
    const int64_t big = std::max(n, m);
    FS_CUDA(sc.get(&ones, (size_t)big));
    FS_CUDA(sc.get(&rows, (size_t)n));
    FS_CUDA(sc.get(&cols, (size_t)m));
    FS_CUDA(sc.get(&partial, kRedMaxBlocks));
    FS_CUDA(sc.get(&res, 2));
    k_fill<<<(unsigned)((big + 255) / 256), 256, 0, s>>>(ones, big, 1.f);
    count_launch();
    FS_CUDA(cudaGetLastError());
    // P 1 and P^T 1 through the plan operators (validation happens there)
    const fs_status st1 = fs_apply_plan(X, a, n, Y, b, m, d, eps, f, g, ones, 1, rows, opt, s);
    if (st1 != FS_OK) return st1;
    const fs_status st2 = fs_apply_plan_t(X, a, n, Y, b, m, d, eps, f, g, ones, 1, cols, opt, s);
    if (st2 != FS_OK) return st2;
    const float *ad, *bd;
    FS_CUDA(sc.device_view(a, (size_t)n, &ad));
    FS_CUDA(sc.device_view(b, (size_t)m, &bd));
    FS_CUDA(reduce_into<1>(rows, ad, n, partial, res, 0, s));
    FS_CUDA(reduce_into<1>(cols, bd, m, partial, res + 1, 0, s));
    FS_CUDA(cudaMemcpyAsync(out, res, 2 * sizeof(double), cudaMemcpyDeviceToHost, s));
    FS_CUDA(cudaStreamSynchronize(s));
    return FS_OK;
}

}  // namespace
}  // namespace fs

extern "C" {

fs_status fs_dual_value(const float* a, int64_t n, const float* b, int64_t m, const float* f,
                        const float* g, double* out, void* stream) {
    try {
        return fs::dual_entry(a, n, b, m, f, g, out, stream);
    } catch (...) {
        return fs::fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_marginal_residuals(const float* X, const float* a, int64_t n, const float* Y,
                                const float* b, int64_t m, int32_t d, float eps, const float* f,
                                const float* g, double* out, const fs_options* opt, void* stream) {
    try {
        return fs::marginal_entry(X, a, n, Y, b, m, d, eps, f, g, out, opt, stream);
    } catch (...) {
        return fs::fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

}  // extern "C"

// Preparation kernels: the common centring shift, packed FMA-path operands,
// squared norms, base-2 log-weights and the bias vector of the first
// half-update ("precomputed log-weight biases" of Proposition 1 in
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 1).
//
// The squared-Euclidean cost is invariant under a common translation of X and
// Y, so both clouds are centred on the mean of all n + m points before the
// dot-product form is used; this keeps |x~|^2 and x~.y~ small and avoids the
// cancellation the dot form would otherwise suffer for far-off clouds.
#include "fs_debug.cuh"
#include "fs_internal.cuh"

namespace fs {

// Block b sums rows [b*R, (b+1)*R) of the concatenation [X; Y] in double,
// one thread per dimension, rows in increasing order.
__global__ void k_colsum(const float* __restrict__ X, int64_t n, const float* __restrict__ Y,
                         int64_t m, int d, int64_t R, double* __restrict__ partial) {
    const int64_t r0 = (int64_t)blockIdx.x * R;
    const int64_t r1 = min(r0 + R, n + m);
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        double s = 0.0;
        for (int64_t r = r0; r < r1; ++r) {
            const bool ok = r < n ? FS_IDX_OK(r * d + k, n * d, 20) : FS_IDX_OK((r - n) * d + k, m * d, 21);
            const float v = !ok ? 0.f : r < n ? X[r * d + k] : Y[(r - n) * d + k];
            s += (double)v;
        }
        partial[(int64_t)blockIdx.x * d + k] = s;
    }
}

__global__ void k_shift_final(const double* __restrict__ partial, int nblk, int d, double inv_total,
                              float* __restrict__ shift) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= d) return;
    double s = 0.0;
    for (int b = 0; b < nblk; ++b) s += partial[(int64_t)b * d + k];
    shift[k] = (float)(s * inv_total);
}

cudaError_t launch_shift(const float* X, int64_t n, const float* Y, int64_t m, int d,
                         double* partial, int nblk_max, float* shift, cudaStream_t s) {
    const int64_t total = n + m;
    int64_t R = (total + nblk_max - 1) / nblk_max;
    if (R < 1) R = 1;
    const int nblk = (int)((total + R - 1) / R);
    const int threads = d >= 256 ? 256 : ((d + 31) / 32) * 32;
    k_colsum<<<nblk, threads, 0, s>>>(X, n, Y, m, d, R, partial);
    k_shift_final<<<(d + 127) / 128, 128, 0, s>>>(partial, nblk, d, 1.0 / (double)total, shift);
    count_launch(2);
    return cudaGetLastError();
}

// One thread per point: centre, zero-pad to D, squared norm, log2 weight, and
// (if `pot` is given) the bias (pot - |p~|^2) L/eps + log2 w in slot D.
template <int D>
__global__ void k_pack_fma(const float* __restrict__ P, const float* __restrict__ w,
                           const float* __restrict__ pot, int64_t rows, int d,
                           const float* __restrict__ shift, float l_over_eps,
                           float* __restrict__ packed, float* __restrict__ norm,
                           float* __restrict__ logw2, const int* __restrict__ perm) {
    constexpr int DS = fma_stride(D);
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows) return;
    const int64_t si = perm != nullptr ? (int64_t)perm[i] : i;
    if (!FS_IDX_OK(si, rows, 22)) return;
    float v[DS];
    float nrm = 0.f;
#pragma unroll
    for (int k = 0; k < DS; ++k) v[k] = 0.f;
#pragma unroll
    for (int k = 0; k < D; ++k) {
        if (k < d) {
            const float c = P[si * d + k] - shift[k];
            v[k] = c;
            nrm = fmaf(c, c, nrm);
        }
    }
    const float lw = log2f(w[si]);
    if (pot != nullptr) v[D] = (pot[si] - nrm) * l_over_eps + lw;
    float4* dst = reinterpret_cast<float4*>(packed + i * DS);
#pragma unroll
    for (int q = 0; q < DS / 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    norm[i] = nrm;
    logw2[i] = lw;
}

cudaError_t launch_pack_fma(const float* P, const float* w, const float* pot, int64_t rows, int d,
                            int D, const float* shift, float l_over_eps, float* packed,
                            float* norm, float* logw2, cudaStream_t s, const int* perm) {
    const int threads = 256;
    const int64_t blocks = (rows + threads - 1) / threads;
    switch (D) {
#define FS_PACK_CASE(DD)                                                                           \
    case DD:                                                                                       \
        k_pack_fma<DD><<<(unsigned)blocks, threads, 0, s>>>(P, w, pot, rows, d, shift, l_over_eps, \
                                                            packed, norm, logw2, perm);            \
        break;
        FS_PACK_CASE(2)
        FS_PACK_CASE(3)
        FS_PACK_CASE(4)
        FS_PACK_CASE(8)
        FS_PACK_CASE(16)
#undef FS_PACK_CASE
        default:
            return cudaErrorInvalidValue;
    }
    count_launch();
    return cudaGetLastError();
}

__global__ void k_scatter_rows(const float* __restrict__ src, const int* __restrict__ perm,
                               int64_t rows, float* __restrict__ dst) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows) return;
    const int64_t di = perm[i];
    if (FS_IDX_OK(di, rows, 23)) dst[di] = src[i];
}

cudaError_t launch_scatter_rows(const float* src, const int* perm, int64_t rows, float* dst,
                                cudaStream_t s) {
    k_scatter_rows<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(src, perm, rows, dst);
    count_launch();
    return cudaGetLastError();
}

FS_BOUNDS_READER(bounds_take_prep)

__global__ void k_phi(const float* __restrict__ f, const float* __restrict__ norm, int64_t n,
                      float l_over_eps, float* __restrict__ phi) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) phi[i] = (f[i] - norm[i]) * l_over_eps;
}

cudaError_t launch_phi(const float* f, const float* norm, int64_t n, float l_over_eps, float* phi,
                       cudaStream_t s) {
    k_phi<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(f, norm, n, l_over_eps, phi);
    count_launch();
    return cudaGetLastError();
}

__global__ void k_count_nonfinite(const float* __restrict__ v, int64_t len,
                                  unsigned int* __restrict__ counter) {
    unsigned int bad = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < len;
         i += (int64_t)gridDim.x * blockDim.x)
        bad += isfinite(v[i]) ? 0u : 1u;
    bad = __reduce_add_sync(0xffffffffu, bad);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(counter, bad);
}

cudaError_t launch_count_nonfinite(const float* v, int64_t len, unsigned int* counter,
                                   cudaStream_t s) {
    int64_t blocks = (len + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    if (blocks < 1) blocks = 1;
    k_count_nonfinite<<<(unsigned)blocks, 256, 0, s>>>(v, len, counter);
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs

// Preparation for the tcgen05 tensor-core path (d > 16): squared norms and
// base-2 log-weights of the centred clouds ("precomputed log-weight biases" of
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 1),
// per-cloud power-of-two scales, the fp16 operand tiles in the exact byte
// order the tensor core reads from shared memory, and the initial biases.
//
// fp16 with a power-of-two scale per cloud keeps an 11-bit significand (the
// precision of TF32) at the f16 MMA rate; the scale cancels exactly in the
// score scale factor kappa 2^-(ex+ey).
#include "fs_tc.cuh"
#include "fs_tc_kernels.cuh"

namespace fs {
namespace tc {

// ---------------------------------------------------------------------------
// preparation

// One warp per point: squared norm of the centred point, log2 of its
// weight, and the running max |coordinate| (as ordered bits, atomicMax).
__global__ void k_stats(const float* __restrict__ P, const float* __restrict__ w, int64_t rows,
                        int d, const float* __restrict__ shift, float* __restrict__ norm,
                        float* __restrict__ logw2, unsigned int* __restrict__ absmax_bits) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float s = 0.f, mx = 0.f;
    const float* p = P + row * d;
    for (int k = lane; k < d; k += 32) {
        const float c = p[k] - shift[k];
        s = fmaf(c, c, s);
        mx = fmaxf(mx, fabsf(c));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
        norm[row] = s;
        logw2[row] = log2f(w[row]);
        atomicMax(absmax_bits, __float_as_uint(mx));
    }
}

// exponent e with max * 2^e in [2^14, 2^15) (0 for an all-zero cloud)
__device__ __forceinline__ int scale_exp(unsigned int bits) {
    const float mx = __uint_as_float(bits);
    if (!(mx > 0.f)) return 0;
    int E;
    frexpf(mx, &E);
    return 15 - E;
}

// params[0] = 2^ex, params[1] = 2^ey, params[2] = kappa 2^-(ex+ey)
__global__ void k_scales(const unsigned int* __restrict__ absmax_bits, float kappa,
                         float* __restrict__ params) {
    const int ex = scale_exp(absmax_bits[0]);
    const int ey = scale_exp(absmax_bits[1]);
    params[0] = ldexpf(1.f, ex);
    params[1] = ldexpf(1.f, ey);
    params[2] = ldexpf(kappa, -(ex + ey));
}

// One thread per 16-byte unit (8 fp16) of the tiled, swizzled operand.  If
// `out_lo` is given it receives the rounding remainder fp16(v - fp16(v)), so
// that hi + lo carries about 22 significant bits.
__global__ void k_to_tiles(const float* __restrict__ P, int64_t rows, int d,
                           const float* __restrict__ shift, const float* __restrict__ scale_ptr,
                           int nch, int64_t row_tiles, uint4* __restrict__ out,
                           uint4* __restrict__ out_lo) {
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t units = row_tiles * BM * nch * 8;
    if (unit >= units) return;
    const int u = (int)(unit & 7);
    const int64_t rowc = unit >> 3;            // (tile, chunk, r) with r fastest
    const int r = (int)(rowc % BM);
    const int64_t tc_ = rowc / BM;
    const int chunk = (int)(tc_ % nch);
    const int64_t tile = tc_ / nch;
    const int64_t row = tile * BM + r;
    const float scale = *scale_ptr;
    const int k0 = chunk * BK + u * 8;
    __align__(16) __half h[8];
    __align__(16) __half l[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int k = k0 + q;
        float v = 0.f;
        if (row < rows && k < d) v = (P[row * d + k] - (shift != nullptr ? shift[k] : 0.f)) * scale;
        h[q] = __float2half_rn(v);
        l[q] = __float2half_rn(v - __half2float(h[q]));
    }
    const int64_t off = (tile * nch + chunk) * (int64_t)CHUNK_BYTES + swz_offset(r, u * 8);
    *reinterpret_cast<uint4*>(reinterpret_cast<char*>(out) + off) = *reinterpret_cast<const uint4*>(h);
    if (out_lo != nullptr)
        *reinterpret_cast<uint4*>(reinterpret_cast<char*>(out_lo) + off) =
            *reinterpret_cast<const uint4*>(l);
}

// bias[j] = (pot_j - norm_j) L/eps + logw2_j for j < rows, -inf for padding;
// with pot == nullptr the real entries are left alone (only padding is set).
__global__ void k_bias_init(const float* __restrict__ pot, const float* __restrict__ norm,
                            const float* __restrict__ logw2, float l_over_eps, int64_t rows,
                            int64_t rows_pad, float* __restrict__ bias) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= rows_pad) return;
    if (j >= rows) bias[j] = -INFINITY;
    else if (pot != nullptr) bias[j] = (pot[j] - norm[j]) * l_over_eps + logw2[j];
}

// Tangent application: one warp per row, crow_i = u_i . x~_i, and the running
// maxima of |u_i|^2 (bits[0]) and of |u_ik| (bits[1]) as ordered bits.
__global__ void k_tan_rows(const float* __restrict__ U, const float* __restrict__ X, int64_t rows,
                           int d, const float* __restrict__ shift, float* __restrict__ crow,
                           unsigned int* __restrict__ bits) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float c = 0.f, s = 0.f, mx = 0.f;
    for (int k = lane; k < d; k += 32) {
        const float u = U[row * d + k];
        c = fmaf(u, X[row * d + k] - shift[k], c);
        s = fmaf(u, u, s);
        mx = fmaxf(mx, fabsf(u));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        c += __shfl_xor_sync(0xffffffffu, c, o);
        s += __shfl_xor_sync(0xffffffffu, s, o);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
        crow[row] = c;
        atomicMax(bits, __float_as_uint(s));
        atomicMax(bits + 1, __float_as_uint(mx));
    }
}

// tparams from bits = (max |u|^2, max |u_k|, max |x~|^2, max |y~|^2) and the
// column cloud's tile scale 2^ey (yscale): |t_ij| <= |u_i| (|y~_j| + |x~_i|)
// = B, and the plan entries p t (|p| <= 1) are carried as p t 2^et with
// B 2^et <= 2^14 in the fp16 plan tile.
//   [0] = 2^-(eu + ey) 2^et   (U K^T accumulator -> t 2^et)
//   [1] = 2^et,  [2] = 2^-et,  [3] = 2^eu (tile scale of U)
__global__ void k_tan_params(const unsigned int* __restrict__ bits, const float* __restrict__ yscale,
                             float* __restrict__ tparams) {
    const int eu = scale_exp(bits[1]);
    const float bound = sqrtf(__uint_as_float(bits[0])) *
                        (sqrtf(__uint_as_float(bits[2])) + sqrtf(__uint_as_float(bits[3])));
    int et = 0;
    if (bound > 0.f && isfinite(bound)) {
        int E;
        frexpf(bound, &E);                 // bound < 2^E
        et = min(max(14 - E, -120), 120);
    }
    tparams[0] = ldexpf(1.f / *yscale, et - eu);
    tparams[1] = ldexpf(1.f, et);
    tparams[2] = ldexpf(1.f, -et);
    tparams[3] = ldexpf(1.f, eu);
}

cudaError_t launch_tan_rows(const float* U, const float* X, int64_t rows, int d, const float* shift,
                            float* crow, unsigned int* bits, cudaStream_t s) {
    const int64_t threads = rows * 32;
    k_tan_rows<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(U, X, rows, d, shift, crow, bits);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_tan_params(const unsigned int* bits, const float* yscale, float* tparams,
                              cudaStream_t s) {
    k_tan_params<<<1, 1, 0, s>>>(bits, yscale, tparams);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_prep_side(const float* P, const float* w, int64_t rows, int d,
                             const float* shift, float* norm, float* logw2,
                             unsigned int* absmax_bits, cudaStream_t s) {
    const int64_t threads = rows * 32;
    k_stats<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(P, w, rows, d, shift, norm, logw2,
                                                              absmax_bits);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_scales(const unsigned int* absmax_bits, float kappa, float* params,
                          cudaStream_t s) {
    k_scales<<<1, 1, 0, s>>>(absmax_bits, kappa, params);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_to_tiles(const float* P, int64_t rows, int d, const float* shift,
                            const float* scale_ptr, int nch, int64_t row_tiles, void* out,
                            void* out_lo, cudaStream_t s) {
    const int64_t units = row_tiles * BM * nch * 8;
    k_to_tiles<<<(unsigned)((units + 255) / 256), 256, 0, s>>>(P, rows, d, shift, scale_ptr, nch,
                                                               row_tiles, (uint4*)out,
                                                               (uint4*)out_lo);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_bias_init(const float* pot, const float* norm, const float* logw2,
                             float l_over_eps, int64_t rows, int64_t rows_pad, float* bias,
                             cudaStream_t s) {
    k_bias_init<<<(unsigned)((rows_pad + 255) / 256), 256, 0, s>>>(pot, norm, logw2, l_over_eps,
                                                                   rows, rows_pad, bias);
    count_launch();
    return cudaGetLastError();
}
}  // namespace tc
}  // namespace fs

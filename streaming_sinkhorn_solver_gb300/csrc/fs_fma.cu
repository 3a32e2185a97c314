// FP32-FMA path for small dimension (d <= 16).
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 2
// (streaming kernels and tiling): the n x m score matrix is never stored;
// each thread keeps its rows resident in registers (row-stationary), the
// block streams the other side's packed (coordinates, bias) records through
// shared memory, the row max and sum-exp are kept on chip (online LSE), and
// the potential and next bias are written back by the same kernel.
//
// At d <= 16 the scores are a handful of FMAs per pair, so the exponential
// (MUFU ex2) and FP32 issue rate bound this path, not memory or tensor cores.
// Scores stay in base 2 (the factor 2 log2(e)/eps is folded into the row
// operand once), so every pair costs exactly one ex2.
#include "fs_internal.cuh"

namespace fs {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 512;   // columns staged in shared memory per pass
constexpr int kGroup = 8;     // columns scored before one max/rescale check

template <int D>
__device__ __forceinline__ void load_cols(const float4* __restrict__ sc, int j, float (&c)[D + 1]) {
    constexpr int DS = fma_stride(D);
    const float4* p = sc + j * (DS / 4);
    float t[DS];
#pragma unroll
    for (int q = 0; q < DS / 4; ++q) {
        const float4 v = p[q];
        t[4 * q] = v.x; t[4 * q + 1] = v.y; t[4 * q + 2] = v.z; t[4 * q + 3] = v.w;
    }
#pragma unroll
    for (int k = 0; k <= D; ++k) c[k] = t[k];
}

template <int D, int RPT>
__global__ void __launch_bounds__(kThreads) k_half_fma(HalfArgs a) {
    constexpr int DS = fma_stride(D);
    __shared__ float4 sc[kChunk * DS / 4];

    const int tid = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * (kThreads * RPT);
    const int64_t c0 = (int64_t)blockIdx.y * a.cols_per_split;
    const int64_t c1 = min(a.nc, c0 + a.cols_per_split);

    float q[RPT][D], M[RPT], S[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        int64_t row = row0 + tid + r * kThreads;
        row = row < a.nr ? row : a.nr - 1;
#pragma unroll
        for (int k = 0; k < D; ++k) q[r][k] = a.rows[row * DS + k] * a.kappa;
        M[r] = -INFINITY;
        S[r] = 0.f;
    }

    for (int64_t cb = c0; cb < c1; cb += kChunk) {
        const int ncol = (int)min((int64_t)kChunk, c1 - cb);
        __syncthreads();
        const float4* src = reinterpret_cast<const float4*>(a.cols + cb * DS);
        for (int e = tid; e < ncol * (DS / 4); e += kThreads) sc[e] = src[e];
        __syncthreads();

        int j = 0;
        for (; j + kGroup <= ncol; j += kGroup) {
            float s[RPT][kGroup];
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                float c[D + 1];
                load_cols<D>(sc, j + u, c);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    float acc = c[D];
#pragma unroll
                    for (int k = 0; k < D; ++k) acc = fmaf(q[r][k], c[k], acc);
                    s[r][u] = acc;
                }
            }
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                float mx = s[r][0];
#pragma unroll
                for (int u = 1; u < kGroup; ++u) mx = fmaxf(mx, s[r][u]);
                if (mx > M[r]) {
                    S[r] *= ex2(M[r] - mx);
                    M[r] = mx;
                }
                float acc = 0.f;
#pragma unroll
                for (int u = 0; u < kGroup; ++u) acc += ex2(s[r][u] - M[r]);
                S[r] += acc;
            }
        }
        for (; j < ncol; ++j) {
            float c[D + 1];
            load_cols<D>(sc, j, c);
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                float acc = c[D];
#pragma unroll
                for (int k = 0; k < D; ++k) acc = fmaf(q[r][k], c[k], acc);
                if (acc > M[r]) {
                    S[r] *= ex2(M[r] - acc);
                    M[r] = acc;
                }
                S[r] += ex2(acc - M[r]);
            }
        }
    }

#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int64_t row = row0 + tid + r * kThreads;
        if (row >= a.nr) continue;
        if (a.splits > 1) {
            a.partial[(int64_t)blockIdx.y * a.nr + row] = make_float2(M[r], S[r]);
        } else {
            const float lse2 = M[r] + log2f(S[r]);
            a.pot[row] = a.rnorm[row] - a.eps_ln2 * lse2;
            a.rows[row * DS + D] = a.rlogw2[row] - lse2;
        }
    }
}

template <int D>
cudaError_t launch_half_fma_t(const HalfArgs& a, cudaStream_t s) {
    constexpr int RPT = D <= 4 ? 4 : (D <= 8 ? 2 : 1);
    const int64_t rows_per_block = (int64_t)kThreads * RPT;
    dim3 grid((unsigned)((a.nr + rows_per_block - 1) / rows_per_block), (unsigned)a.splits);
    k_half_fma<D, RPT><<<grid, kThreads, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

__global__ void k_merge_lse(const float2* __restrict__ partial, int splits, int64_t nr,
                            const float* __restrict__ rnorm, const float* __restrict__ rlogw2,
                            float eps_ln2, float* __restrict__ pot, float* __restrict__ bias,
                            int64_t bias_stride) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nr) return;
    float M = -INFINITY;
    for (int sp = 0; sp < splits; ++sp) M = fmaxf(M, partial[(int64_t)sp * nr + i].x);
    float S = 0.f;
    for (int sp = 0; sp < splits; ++sp) {
        const float2 p = partial[(int64_t)sp * nr + i];
        if (p.x != -INFINITY) S += p.y * ex2(p.x - M);   // a padding-only split adds nothing
    }
    const float lse2 = M + log2f(S);
    if (rnorm == nullptr) {  // log2-sum-exp only (pre-pass of plan application)
        pot[i] = lse2;
        return;
    }
    pot[i] = rnorm[i] - eps_ln2 * lse2;
    bias[i * bias_stride] = rlogw2[i] - lse2;
}

// ---------------------------------------------------------------------------
// Plan application (Method 3): out_i = sum_j P_ij V_j with
//   P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps) = a_i 2^{phi_i} 2^{s_ij},
// phi_i = (f_i - |x~_i|^2) L/eps and s_ij the f-update score built from g.
// Each thread owns one row and KC columns of V; a running max M keeps the
// accumulator O = sum_j 2^{s_ij - M} V_j in range, so out_i = a_i 2^{phi_i+M} O.

constexpr int kApplyThreads = 128;
constexpr int kApplyChunk = 256;

template <int D, int KC>
__global__ void __launch_bounds__(kApplyThreads) k_apply_fma(ApplyArgs a) {
    constexpr int DS = fma_stride(D);
    __shared__ float4 sc[kApplyChunk * DS / 4];
    __shared__ float sv[kApplyChunk * KC];

    const int tid = threadIdx.x;
    const int64_t row = (int64_t)blockIdx.x * kApplyThreads + tid;
    const int64_t rr = row < a.n ? row : a.n - 1;
    const int64_t c0 = (int64_t)blockIdx.y * a.cols_per_split;
    const int64_t c1 = min(a.m, c0 + a.cols_per_split);
    const int kc0 = blockIdx.z * KC;
    const int kw = min(KC, a.k - kc0);

    float q[D];
#pragma unroll
    for (int k = 0; k < D; ++k) q[k] = a.rows[rr * DS + k] * a.kappa;
    float M = -INFINITY;
    float O[KC];
#pragma unroll
    for (int c = 0; c < KC; ++c) O[c] = 0.f;

    for (int64_t cb = c0; cb < c1; cb += kApplyChunk) {
        const int ncol = (int)min((int64_t)kApplyChunk, c1 - cb);
        __syncthreads();
        const float4* src = reinterpret_cast<const float4*>(a.cols + cb * DS);
        for (int e = tid; e < ncol * (DS / 4); e += kApplyThreads) sc[e] = src[e];
        for (int e = tid; e < ncol * KC; e += kApplyThreads) {
            const int j = e / KC, c = e - j * KC;
            sv[e] = c < kw ? a.V[(cb + j) * a.k + kc0 + c] : 0.f;
        }
        __syncthreads();
        for (int j = 0; j < ncol; ++j) {
            float cv[D + 1];
            load_cols<D>(sc, j, cv);
            float sij = cv[D];
#pragma unroll
            for (int k = 0; k < D; ++k) sij = fmaf(q[k], cv[k], sij);
            if (sij > M) {
                const float r = ex2(M - sij);
#pragma unroll
                for (int c = 0; c < KC; ++c) O[c] *= r;
                M = sij;
            }
            const float p = ex2(sij - M);
#pragma unroll
            for (int c = 0; c < KC; ++c) O[c] = fmaf(p, sv[j * KC + c], O[c]);
        }
    }
    if (row >= a.n) return;
    if (a.splits > 1) {
        const int64_t base = ((int64_t)blockIdx.y * a.n + row) * (a.k + 1);
        if (blockIdx.z == 0) a.partial[base] = M;
        for (int c = 0; c < kw; ++c) a.partial[base + 1 + kc0 + c] = O[c];
        return;
    }
    const float w = exp2f(a.phi[row] + M);
    for (int c = 0; c < kw; ++c) {
        const float t = w * O[c];
        float o;
        if (a.mode == APPLY_PV) o = a.a[row] * t;
        else if (a.mode == APPLY_BARY) o = t;
        else o = 2.f * a.a[row] * (a.X[row * a.d + kc0 + c] - t);
        a.out[row * a.k + kc0 + c] = o;
    }
}

template <int D>
cudaError_t launch_apply_fma_t(const ApplyArgs& a, cudaStream_t s) {
    const unsigned kchunks16 = (unsigned)((a.k + 15) / 16);
    dim3 grid((unsigned)((a.n + kApplyThreads - 1) / kApplyThreads), (unsigned)a.splits);
    if (a.k <= 4) {
        grid.z = 1;
        k_apply_fma<D, 4><<<grid, kApplyThreads, 0, s>>>(a);
    } else {
        grid.z = kchunks16;
        k_apply_fma<D, 16><<<grid, kApplyThreads, 0, s>>>(a);
    }
    count_launch();
    return cudaGetLastError();
}

__global__ void k_merge_apply(ApplyArgs a) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.n) return;
    const int64_t stride = (int64_t)a.n * (a.k + 1);
    float M = -INFINITY;
    for (int sp = 0; sp < a.splits; ++sp) M = fmaxf(M, a.partial[sp * stride + i * (a.k + 1)]);
    const float w = exp2f(a.phi[i] + M);
    for (int c = 0; c < a.k; ++c) {
        float O = 0.f;
        for (int sp = 0; sp < a.splits; ++sp) {
            const float* p = a.partial + sp * stride + i * (a.k + 1);
            O += p[1 + c] * ex2(p[0] - M);
        }
        const float t = w * O;
        float o;
        if (a.mode == APPLY_PV) o = a.a[i] * t;
        else if (a.mode == APPLY_BARY) o = t;
        else o = 2.f * a.a[i] * (a.X[i * a.d + c] - t);
        a.out[i * a.k + c] = o;
    }
}

}  // namespace

cudaError_t launch_half_fma(int D, const HalfArgs& a, cudaStream_t s) {
    switch (D) {
        case 2: return launch_half_fma_t<2>(a, s);
        case 3: return launch_half_fma_t<3>(a, s);
        case 4: return launch_half_fma_t<4>(a, s);
        case 8: return launch_half_fma_t<8>(a, s);
        case 16: return launch_half_fma_t<16>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge_lse(const float2* partial, int splits, int64_t nr, const float* rnorm,
                             const float* rlogw2, float eps_ln2, float* pot, float* bias,
                             int64_t bias_stride, cudaStream_t s) {
    k_merge_lse<<<(unsigned)((nr + 255) / 256), 256, 0, s>>>(partial, splits, nr, rnorm, rlogw2,
                                                             eps_ln2, pot, bias, bias_stride);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_apply_fma(int D, const ApplyArgs& a, cudaStream_t s) {
    switch (D) {
        case 2: return launch_apply_fma_t<2>(a, s);
        case 3: return launch_apply_fma_t<3>(a, s);
        case 4: return launch_apply_fma_t<4>(a, s);
        case 8: return launch_apply_fma_t<8>(a, s);
        case 16: return launch_apply_fma_t<16>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge_apply(const ApplyArgs& a, cudaStream_t s) {
    k_merge_apply<<<(unsigned)((a.n + 127) / 128), 128, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs

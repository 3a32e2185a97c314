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
#include "fs_debug.cuh"
#include "fs_internal.cuh"

#include <cooperative_groups.h>

#include <algorithm>
#include <type_traits>

namespace fs {

namespace {

constexpr int kThreads = 256;
constexpr int kGroup = 8;     // columns scored per max check

// Guarded range of a row's sum S = sum_j 2^{s_ij - M_ref} when the offset is
// the previous LSE instead of the running max: below 2^-64 the terms that
// underflowed could matter, above 2^126 the sum could overflow.  Outside the
// range the row is recomputed with the online max.
constexpr float kMinRefSum = 5.421010862427522e-20f;   // 2^-64
constexpr float kMaxRefSum = 8.507059173023462e+37f;   // 2^126

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

// Shared-memory column records are stored duplicated, (y0, y0, y1, y1, ...,
// bias, bias), so that one packed fma.rn.f32x2 scores a column against two
// rows at once with no register shuffling.
__host__ __device__ constexpr int fma_dup_stride(int D) { return (2 * (D + 1) + 3) / 4 * 4; }
__host__ __device__ constexpr int fma_chunk(int D) { return D <= 4 ? 512 : 256; }

// max(m, v[0], ..., v[G-1]) as a depth-2 tree of 3-input maxima.
template <int G>
__device__ __forceinline__ float max_tree(const float (&v)[G], float m) {
    static_assert(G == 1 || G == 8, "group sizes 1 and 8");
    if constexpr (G == 1) {
        return fmaxf(m, v[0]);
    } else {
        return max3(max3(v[0], v[1], v[2]), max3(v[3], v[4], v[5]), max3(v[6], v[7], m));
    }
}

// A row's reference M moves only when its max exceeds M by more than this
// (log2 units), so terms 2^{s - M} stay below 2^8 and the rescale is rare.
constexpr float kMaxSlack = 8.f;

// Scores of G columns (shared records j .. j+G-1) against RP row pairs.
template <int D, int RP, int G>
__device__ __forceinline__ void fma_scores(const float4* __restrict__ sc, int j,
                                           const uint64_t (&q)[RP][D], uint64_t (&s)[RP][G]) {
    constexpr int DD = fma_dup_stride(D);
#pragma unroll
    for (int u = 0; u < G; ++u) {
        const float4* p = sc + (j + u) * (DD / 4);
        uint64_t c[DD / 2];
#pragma unroll
        for (int w = 0; w < DD / 4; ++w) {
            const float4 v = p[w];
            c[2 * w] = pk(v.x, v.y);
            c[2 * w + 1] = pk(v.z, v.w);
        }
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            uint64_t acc = c[D];
#pragma unroll
            for (int k = 0; k < D; ++k) acc = fma2(q[r][k], c[k], acc);
            s[r][u] = acc;
        }
    }
}

// S[r] += sum_u 2^{s[r][u] - M} (nm = packed -M), summed as a tree.
template <int RP, int G>
__device__ __forceinline__ void fma_sum_exp(const uint64_t (&s)[RP][G], const uint64_t (&nm)[RP],
                                            uint64_t (&S)[RP]) {
#pragma unroll
    for (int r = 0; r < RP; ++r) {
        uint64_t e[G];
#pragma unroll
        for (int u = 0; u < G; ++u) {
            float x0, x1;
            upk(add2(s[r][u], nm[r]), x0, x1);
            e[u] = pk(ex2(x0), ex2(x1));
        }
#pragma unroll
        for (int w = 1; w < G; w *= 2) {
#pragma unroll
            for (int u = 0; u + w < G; u += 2 * w) e[u] = add2(e[u], e[u + w]);
        }
        S[r] = add2(S[r], e[0]);
    }
}

// S[r] += sum_u 2^{s[r][u]}: the scores already carry the row offset (folded
// into the staged column records).
template <int RP, int G>
__device__ __forceinline__ void fma_sum_exp_noff(const uint64_t (&s)[RP][G], uint64_t (&S)[RP]) {
#pragma unroll
    for (int r = 0; r < RP; ++r) {
        uint64_t e[G];
#pragma unroll
        for (int u = 0; u < G; ++u) {
            float x0, x1;
            upk(s[r][u], x0, x1);
            e[u] = pk(ex2(x0), ex2(x1));
        }
#pragma unroll
        for (int w = 1; w < G; w *= 2) {
#pragma unroll
            for (int u = 0; u + w < G; u += 2 * w) e[u] = add2(e[u], e[u + w]);
        }
        S[r] = add2(S[r], e[0]);
    }
}

// Sum of NV values over the CTA, the same bits in every thread: warp
// butterflies, then the warps' sums in warp order (red: NV * (warps + 1)).
template <int NV>
__device__ __forceinline__ void cta_sum(float (&v)[NV], float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int W = kThreads / 32;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int o = 16; o; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    if (lane == 0)
#pragma unroll
        for (int k = 0; k < NV; ++k) red[warp * NV + k] = v[k];
    __syncthreads();
    if (threadIdx.x < NV) {
        float t = 0.f;
        for (int w = 0; w < W; ++w) t += red[w * NV + threadIdx.x];
        red[W * NV + threadIdx.x] = t;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < NV; ++k) v[k] = red[W * NV + k];
    __syncthreads();
}

// Folded offsets (rows in Morton order).  The CTA fits its rows' previous
// LSEs M_i by an affine function of their kappa-scaled coordinates q_i,
// A_i = mu + h . q_i (least squares; a D x D Cholesky solve, h = 0 when
// singular), with mu raised so the largest residual M_i - A_i is kFoldTop.
// Staging the columns as (y - h, bias - mu) makes the score chain yield
// s_ij - A_i.  Sums relative to A_i stay in the guarded range while the
// residuals spread less than kFoldSpread; a CTA whose rows spread more keeps
// the per-row offsets (fold = false).  fit[0 .. D-1] = h, fit[D] = mu.
constexpr float kFoldTop = 80.f;
constexpr float kFoldSpread = 130.f;

template <int D, int RPT>
__device__ __forceinline__ bool cta_offset_fit(const float (&qv)[RPT][D], const float (&M)[RPT],
                                               const bool (&valid)[RPT], float* red, float* fit) {
    float m1[D + 2];
#pragma unroll
    for (int k = 0; k < D + 2; ++k) m1[k] = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        if (!valid[i]) continue;
        m1[0] += 1.f;
        m1[1] += M[i];
#pragma unroll
        for (int k = 0; k < D; ++k) m1[2 + k] += qv[i][k];
    }
    cta_sum<D + 2>(m1, red);
    const float inv_n = 1.f / m1[0];
    const float mbar = m1[1] * inv_n;
    float qbar[D];
#pragma unroll
    for (int k = 0; k < D; ++k) qbar[k] = m1[2 + k] * inv_n;
    constexpr int NC = D * (D + 1) / 2;
    float m2[NC + D];
#pragma unroll
    for (int k = 0; k < NC + D; ++k) m2[k] = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        if (!valid[i]) continue;
        const float dm = M[i] - mbar;
        int t = 0;
#pragma unroll
        for (int k = 0; k < D; ++k) {
            const float dk = qv[i][k] - qbar[k];
            m2[NC + k] += dk * dm;
#pragma unroll
            for (int l = k; l < D; ++l) m2[t++] += dk * (qv[i][l] - qbar[l]);
        }
    }
    cta_sum<NC + D>(m2, red);
    float C[D][D], c[D], h[D];
    {
        int t = 0;
        float tr = 0.f;
#pragma unroll
        for (int k = 0; k < D; ++k) {
            c[k] = m2[NC + k];
#pragma unroll
            for (int l = k; l < D; ++l) {
                C[k][l] = C[l][k] = m2[t++];
            }
            tr += C[k][k];
        }
        const float lam = 1e-4f * tr / D + 1e-30f;
#pragma unroll
        for (int k = 0; k < D; ++k) C[k][k] += lam;
    }
    bool ok = true;
#pragma unroll
    for (int k = 0; k < D; ++k) {
#pragma unroll
        for (int l = 0; l < k; ++l) C[k][k] -= C[k][l] * C[k][l];
        ok = ok && C[k][k] > 0.f;
        C[k][k] = sqrtf(fmaxf(C[k][k], 1e-30f));
#pragma unroll
        for (int r = k + 1; r < D; ++r) {
#pragma unroll
            for (int l = 0; l < k; ++l) C[r][k] -= C[r][l] * C[k][l];
            C[r][k] /= C[k][k];
        }
    }
#pragma unroll
    for (int k = 0; k < D; ++k) {
#pragma unroll
        for (int l = 0; l < k; ++l) c[k] -= C[k][l] * c[l];
        c[k] /= C[k][k];
    }
#pragma unroll
    for (int k = D - 1; k >= 0; --k) {
#pragma unroll
        for (int l = k + 1; l < D; ++l) c[k] -= C[l][k] * h[l];
        h[k] = c[k] / C[k][k];
        ok = ok && isfinite(h[k]);
    }
    if (!ok) {
#pragma unroll
        for (int k = 0; k < D; ++k) h[k] = 0.f;
    }
    float mu = mbar;
#pragma unroll
    for (int k = 0; k < D; ++k) mu -= h[k] * qbar[k];
    // residual range over the CTA (max of r and of -r)
    float rr[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        if (!valid[i]) continue;
        float a = mu;
#pragma unroll
        for (int k = 0; k < D; ++k) a = fmaf(h[k], qv[i][k], a);
        rr[0] = fmaxf(rr[0], M[i] - a);
        rr[1] = fmaxf(rr[1], a - M[i]);
    }
    {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        constexpr int W = kThreads / 32;
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int o = 16; o; o >>= 1) rr[k] = fmaxf(rr[k], __shfl_xor_sync(0xffffffffu, rr[k], o));
        if (lane == 0) {
            red[2 * warp] = rr[0];
            red[2 * warp + 1] = rr[1];
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float a = -INFINITY, b = -INFINITY;
            for (int w = 0; w < W; ++w) {
                a = fmaxf(a, red[2 * w]);
                b = fmaxf(b, red[2 * w + 1]);
            }
            const bool fold = a + b <= kFoldSpread && isfinite(a + b);
#pragma unroll
            for (int k = 0; k < D; ++k) fit[k] = h[k];
            fit[D] = mu + a - kFoldTop;
            fit[D + 1] = fold ? 1.f : 0.f;
        }
        __syncthreads();
    }
    return fit[D + 1] != 0.f;
}

// Online fold of G scores per row into (M, S): S = sum 2^{s - M}.  Mt = M +
// slack is the threshold a new max must pass to move M; nm holds the packed
// -M of each row pair.  The check is warp-uniform, so the rescale branch
// never diverges.
template <int RP, int G>
__device__ __forceinline__ void fma_fold(const uint64_t (&s)[RP][G], float (&M)[2 * RP],
                                         float (&Mt)[2 * RP], uint64_t (&nm)[RP],
                                         uint64_t (&S)[RP]) {
    float m[2 * RP];
    bool grow = false;
#pragma unroll
    for (int r = 0; r < RP; ++r) {
        float lo[G], hi[G];
#pragma unroll
        for (int u = 0; u < G; ++u) upk(s[r][u], lo[u], hi[u]);
        m[2 * r] = max_tree<G>(lo, Mt[2 * r]);
        m[2 * r + 1] = max_tree<G>(hi, Mt[2 * r + 1]);
        grow |= (m[2 * r] > Mt[2 * r]) | (m[2 * r + 1] > Mt[2 * r + 1]);
    }
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int i = 0; i < 2 * RP; ++i) {
            const float n = m[i] > Mt[i] ? m[i] : M[i];
            m[i] = ex2(M[i] - n);   // rescale factor (1 where M stays)
            M[i] = n;
            Mt[i] = n + kMaxSlack;
        }
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            S[r] = fma2(S[r], pk(m[2 * r], m[2 * r + 1]), pk(0.f, 0.f));
            nm[r] = pk(-M[2 * r], -M[2 * r + 1]);
        }
    }
    fma_sum_exp<RP, G>(s, nm, S);
}

// Append `row` to the list of rows the fixup kernel recomputes.
__device__ __forceinline__ void push_fix(const HalfArgs& a, int64_t row) {
    const unsigned int slot = atomicAdd(&a.fix_count[0], 1u);
    if (slot < (unsigned int)a.nr) a.fix_list[slot] = (int)row;
}

// Half-update, RP row pairs per thread (rows row0 + tid + i * kThreads,
// i < 2 RP).  MODE 0: online max.  MODE 1: each row's offset is the LSE of
// its previous half-update, log2 w_i - (bias slot), so no max is tracked;
// the sum is range-checked at the end (here when the split is the whole row,
// else in the merge).  MODE 2: as 1, through the CTA's affine fit of those
// LSEs folded into the staged columns (cta_offset_fit; rows in Morton order).
// The work of one CTA: row block rb (rows rb * 512 RP + ...) against the
// columns of split sp.
template <int D, int RP, int MODE>
__device__ __forceinline__ void half_body(const HalfArgs& a, int64_t rb, int64_t sp) {
    constexpr bool REF = MODE >= 1;
    constexpr int DS = fma_stride(D);
    constexpr int DD = fma_dup_stride(D);
    constexpr int CH = fma_chunk(D);
    constexpr int RPT = 2 * RP;
    __shared__ float4 sc[CH * DD / 4];
    __shared__ float fit[D + 2];

    const int tid = threadIdx.x;
    const int64_t row0 = rb * (kThreads * RPT);
    const int64_t c0 = sp * a.cols_per_split;
    const int64_t c1 = min(a.nc, c0 + a.cols_per_split);

    uint64_t q[RP][D];
    float M[RPT], Mt[RPT];
    uint64_t S[RP], nm[RP];
#pragma unroll
    for (int r = 0; r < RP; ++r) {
        int64_t ra = row0 + tid + (2 * r) * kThreads, rb = ra + kThreads;
        ra = ra < a.nr ? ra : a.nr - 1;
        rb = rb < a.nr ? rb : a.nr - 1;
#pragma unroll
        for (int k = 0; k < D; ++k)
            q[r][k] = pk(a.rows[ra * DS + k] * a.kappa, a.rows[rb * DS + k] * a.kappa);
        if (REF) {
            M[2 * r] = a.rlogw2[ra] - a.rows[ra * DS + D];
            M[2 * r + 1] = a.rlogw2[rb] - a.rows[rb * DS + D];
        } else {
            M[2 * r] = M[2 * r + 1] = -INFINITY;
        }
        Mt[2 * r] = Mt[2 * r + 1] = -INFINITY;
        S[r] = pk(0.f, 0.f);
        nm[r] = REF ? pk(-M[2 * r], -M[2 * r + 1]) : pk(INFINITY, INFINITY);
    }
    // MODE 2: the CTA fits its rows' previous LSEs (every column split of a
    // row block computes the same fit from the same values): h, mu and
    // whether the fit holds, in fit[]; the rows' offsets become the fitted A_i
    bool fold = false;
    if constexpr (MODE == 2) {
        __shared__ float red[(D * (D + 1) / 2 + D) * (kThreads / 32 + 1)];
        float qv[RPT][D];
        bool valid[RPT];
#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
            for (int k = 0; k < D; ++k) upk(q[r][k], qv[2 * r][k], qv[2 * r + 1][k]);
#pragma unroll
        for (int i = 0; i < RPT; ++i) valid[i] = row0 + tid + i * kThreads < a.nr;
        fold = cta_offset_fit<D, RPT>(qv, M, valid, red, fit);
        if (fold) {
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                float A = fit[D];
#pragma unroll
                for (int k = 0; k < D; ++k) A = fmaf(fit[k], qv[i][k], A);
                M[i] = A;
            }
        }
    }

    float* sf = reinterpret_cast<float*>(sc);
    // the column sweep; FOLD: the staged records carry the CTA's fit and the
    // scores the row offsets (two copies of the loop, so that the folded one
    // keeps no per-row offsets live)
    auto sweep = [&](auto fold_tag) {
        constexpr bool FOLD = decltype(fold_tag)::value;
        for (int64_t cb = c0; cb < c1; cb += CH) {
            const int ncol = (int)min((int64_t)CH, c1 - cb);
            __syncthreads();
            // stage (coordinates, bias) records, each value written twice
            for (int e = tid; e < ncol * (D + 1); e += kThreads) {
                const int jj = e / (D + 1), k = e - jj * (D + 1);
                const int64_t src = (cb + jj) * DS + k;
                float v = FS_IDX_OK(src, a.nc * DS, 1) ? a.cols[src] : 0.f;
                if (FOLD) v -= fit[k];   // coordinates minus h, bias minus mu
                sf[jj * DD + 2 * k] = v;
                sf[jj * DD + 2 * k + 1] = v;
            }
            __syncthreads();
            int j = 0;
            for (; j + kGroup <= ncol; j += kGroup) {
                uint64_t s[RP][kGroup];
                fma_scores<D, RP, kGroup>(sc, j, q, s);
                if (FOLD) fma_sum_exp_noff<RP, kGroup>(s, S);
                else if (REF) fma_sum_exp<RP, kGroup>(s, nm, S);
                else fma_fold<RP, kGroup>(s, M, Mt, nm, S);
            }
            for (; j < ncol; ++j) {
                uint64_t s[RP][1];
                fma_scores<D, RP, 1>(sc, j, q, s);
                if (FOLD) fma_sum_exp_noff<RP, 1>(s, S);
                else if (REF) fma_sum_exp<RP, 1>(s, nm, S);
                else fma_fold<RP, 1>(s, M, Mt, nm, S);
            }
        }
    };
    if (MODE == 2 && fold) sweep(std::true_type{});
    else sweep(std::false_type{});

    float Sf[RPT];
#pragma unroll
    for (int r = 0; r < RP; ++r) upk(S[r], Sf[2 * r], Sf[2 * r + 1]);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int64_t row = row0 + tid + i * kThreads;
        if (row >= a.nr) continue;
        if (a.splits > 1) {
            const int64_t pi = sp * a.nr + row;
            if (FS_IDX_OK(pi, (int64_t)a.splits * a.nr, 2)) a.partial[pi] = make_float2(M[i], Sf[i]);
        } else {
            if (REF && !(Sf[i] >= kMinRefSum && Sf[i] <= kMaxRefSum)) push_fix(a, row);
            const float lse2 = M[i] + log2f(Sf[i]);
            a.pot[row] = a.rnorm[row] - a.eps_ln2 * lse2;
            a.rows[row * DS + D] = a.rlogw2[row] - lse2;
        }
    }
}

// Four CTAs per SM in the folded mode (64 registers; measured 1.4 % faster
// than three at d = 3), three (d <= 8) or two otherwise.
template <int D, int RP, int MODE>
__global__ void __launch_bounds__(kThreads, MODE == 2 ? 4 : D <= 8 ? 3 : 2) k_half_fma(HalfArgs a) {
    half_body<D, RP, MODE>(a, blockIdx.x, blockIdx.y);
}

template <int D>
cudaError_t launch_half_fma_t(const HalfArgs& a, cudaStream_t s) {
    constexpr int RP = fma_row_pairs(D);
    const int64_t rows_per_block = (int64_t)kThreads * 2 * RP;
    static_assert(kThreads * 2 * RP == fma_rows_per_block(D), "row blocking");
    dim3 grid((unsigned)((a.nr + rows_per_block - 1) / rows_per_block), (unsigned)a.splits);
    bool launched = false;
    if constexpr (D <= 4) {
        if (a.use_ref == 2) {
            k_half_fma<D, RP, 2><<<grid, kThreads, 0, s>>>(a);
            launched = true;
        }
    }
    if (!launched) {
        if (a.use_ref) k_half_fma<D, RP, 1><<<grid, kThreads, 0, s>>>(a);
        else k_half_fma<D, RP, 0><<<grid, kThreads, 0, s>>>(a);
    }
    count_launch();
    return cudaGetLastError();
}

// (M, S) := the (max, sum) pair of the union: S 2^M + So 2^Mo = S' 2^M'.
__device__ __forceinline__ void merge_pair(float& M, float& S, float Mo, float So) {
    const float Mn = fmaxf(M, Mo);
    S = (M == -INFINITY ? 0.f : S * ex2(M - Mn)) + (Mo == -INFINITY ? 0.f : So * ex2(Mo - Mn));
    M = Mn;
}

// Merge of the column splits' (max, sum) pairs of each row: `lanes` threads
// per row (a power of two up to 32, about the split count), each folding
// the splits l, l + lanes, ... in order, then a butterfly over the row's
// lanes; fixed assignment and order, so the result does not depend on
// timing.  Whole warps run, so that every lane takes part in the shuffles.
__device__ __forceinline__ void merge_slot(int64_t t, const float2* __restrict__ partial, int splits,
                                           int64_t nr, const float* __restrict__ rnorm,
                                           const float* __restrict__ rlogw2, float eps_ln2,
                                           float* __restrict__ pot, float* __restrict__ bias,
                                           int64_t bias_stride, int* __restrict__ fix_list,
                                           unsigned int* __restrict__ fix_count, int lanes) {
    const int64_t i = t / lanes;
    const int l = (int)(t % lanes);
    float M = -INFINITY, S = 0.f;
    if (i < nr) {
        for (int sp = l; sp < splits; sp += lanes) {
            if (!FS_IDX_OK((int64_t)sp * nr + i, (int64_t)splits * nr, 3)) continue;
            const float2 p = partial[(int64_t)sp * nr + i];
            if (p.x != -INFINITY) merge_pair(M, S, p.x, p.y);   // a padding-only split adds nothing
        }
    }
    for (int o = lanes >> 1; o; o >>= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
        const float So = __shfl_xor_sync(0xffffffffu, S, o);
        merge_pair(M, S, Mo, So);
    }
    if (i >= nr || l != 0) return;
    if (fix_list != nullptr && !(S >= kMinRefSum && S <= kMaxRefSum)) {
        const unsigned int slot = atomicAdd(&fix_count[0], 1u);
        if (slot < (unsigned int)nr) fix_list[slot] = (int)i;
    }
    const float lse2 = M + log2f(S);
    if (rnorm == nullptr) {  // log2-sum-exp only (pre-pass of plan application)
        pot[i] = lse2;
        return;
    }
    pot[i] = rnorm[i] - eps_ln2 * lse2;
    bias[i * bias_stride] = rlogw2[i] - lse2;
}

__global__ void k_merge_lse(const float2* __restrict__ partial, int splits, int64_t nr,
                            const float* __restrict__ rnorm, const float* __restrict__ rlogw2,
                            float eps_ln2, float* __restrict__ pot, float* __restrict__ bias,
                            int64_t bias_stride, int* __restrict__ fix_list,
                            unsigned int* __restrict__ fix_count, int lanes) {
    merge_slot((int64_t)blockIdx.x * blockDim.x + threadIdx.x, partial, splits, nr, rnorm, rlogw2,
               eps_ln2, pot, bias, bias_stride, fix_list, fix_count, lanes);
}

// Recompute, with the online max, the rows listed by a guarded half-update:
// one warp per listed row, lanes striding over all columns, then a shuffle
// merge of the lanes' (max, sum).  The list length is read once per block;
// the last block to finish resets the list for the next half-update.
constexpr int kFixBlocks = 64;

// One listed row, by one warp (lane = its lane).
template <int D>
__device__ __forceinline__ void fix_row(const HalfArgs& a, int64_t row, int lane) {
    constexpr int DS = fma_stride(D);
    {
        float q[D];
#pragma unroll
        for (int k = 0; k < D; ++k) q[k] = a.rows[row * DS + k] * a.kappa;
        float M = -INFINITY, S = 0.f;
        for (int64_t j = lane; j < a.nc; j += 32) {
            float s = a.cols[j * DS + D];
#pragma unroll
            for (int k = 0; k < D; ++k) s = fmaf(q[k], a.cols[j * DS + k], s);
            if (s > M) {
                S *= ex2(M - s);
                M = s;
            }
            S += ex2(s - M);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
            const float So = __shfl_xor_sync(0xffffffffu, S, o);
            const float Mn = fmaxf(M, Mo);
            S = (M == -INFINITY ? 0.f : S * ex2(M - Mn)) + (Mo == -INFINITY ? 0.f : So * ex2(Mo - Mn));
            M = Mn;
        }
        if (lane == 0) {
            const float lse2 = M + log2f(S);
            a.pot[row] = a.rnorm[row] - a.eps_ln2 * lse2;
            a.rows[row * DS + D] = a.rlogw2[row] - lse2;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(256) k_fix_fma(HalfArgs a) {
    __shared__ unsigned int s_cnt;
    if (threadIdx.x == 0) s_cnt = min(*(volatile unsigned int*)&a.fix_count[0], (unsigned int)a.nr);
    __syncthreads();
    const unsigned int cnt = s_cnt;
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (unsigned int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < cnt; w += warps) {
        const int64_t row = a.fix_list[w];
        if (!FS_IDX_OK(row, a.nr, 4)) continue;
        fix_row<D>(a, row, lane);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&a.fix_count[1], 1u) == gridDim.x - 1) {
            if (a.fix_stats) {
                a.fix_stats[0] += 1ull;
                a.fix_stats[1] += cnt;
            }
            a.fix_count[0] = 0;
            a.fix_count[1] = 0;
            __threadfence();
        }
    }
}

template <int D>
cudaError_t launch_fix_fma_t(const HalfArgs& a, cudaStream_t s) {
    k_fix_fma<D><<<kFixBlocks, 256, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Whole solve in one cooperative launch, for problems small enough that
// launches dominate (c1, c2 at 10^4 points).  Every half-update runs the same
// three phases as the multi-launch path -- the half-update work items (row
// block, column split), the split merge, the fixup of guarded rows -- with
// the same per-row arithmetic, the same merge order (merge_slot) and the same
// fixup (fix_row), so the potentials are bitwise those of separate launches.
// The phases are separated by a grid barrier (all blocks are co-resident:
// cudaLaunchCooperativeKernel) whose waits give up after SmallArgs::timeout_ns,
// set ERR_TIMEOUT_BARRIER in the error word and end the kernel.
//
// The two sides use separate fixup lists: the f-half's list is reset (and
// counted) by block 0 during the g-half and vice versa, when every block has
// read it and before it is written again.

__device__ __forceinline__ uint64_t fma_globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// bar[0] counts arrivals over the whole launch (zeroed before it): barrier k
// is passed once it reaches k * gridDim.x.  Each block adds one with release
// semantics (after its threads' writes, ordered by the block barrier) and
// polls with acquire loads, so the critical path is the last arrival and one
// poll.  gen counts the barriers this block has passed.  Returns false (in
// every thread) when the wait gave up.
__device__ __forceinline__ bool grid_barrier(unsigned int* bar, unsigned int& gen, uint32_t* err,
                                             uint64_t timeout_ns) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int target = (gen + 1u) * gridDim.x;
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
        int ok = 1;
        const uint64_t deadline = fma_globaltimer() + timeout_ns;
        for (;;) {
            unsigned int v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
            if ((int)(v - target) >= 0) break;
            if (fma_globaltimer() > deadline) {
                atomicOr(err, ERR_TIMEOUT_BARRIER);
                ok = 0;
                break;
            }
            __nanosleep(32);
        }
        s_ok = ok;
    }
    __syncthreads();
    ++gen;
    return s_ok != 0;
}

// The barrier between phases: the grid barrier above, or, when the whole
// grid is one thread-block cluster (at most 16 blocks), the cluster's
// hardware barrier, whose release/acquire orders the blocks' global writes
// and reads like the grid barrier's.
template <bool CLUSTER>
__device__ __forceinline__ bool phase_barrier(const SmallArgs& s, unsigned int& gen) {
    if (CLUSTER) {
        cooperative_groups::this_cluster().sync();
        ++gen;
        return true;
    }
    return grid_barrier(s.bar, gen, s.err, s.timeout_ns);
}

template <int D, int RP, bool CLUSTER>
__global__ void __launch_bounds__(kThreads, 3) k_solve_small(const __grid_constant__ SmallArgs s) {
    unsigned int gen = 0;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    for (int it = 0; it < s.n_iter; ++it) {
        const bool ref = it >= s.ref_from;
        for (int side = 0; side < 2; ++side) {
            const HalfArgs& a = s.h[side];
            const int64_t items = s.row_blocks[side] * a.splits;
            for (int64_t w = blockIdx.x; w < items; w += gridDim.x) {
                const int64_t rb = w % s.row_blocks[side], sp = w / s.row_blocks[side];
                if (ref) half_body<D, RP, 1>(a, rb, sp);
                else half_body<D, RP, 0>(a, rb, sp);
            }
            if (a.splits > 1) {
                if (!phase_barrier<CLUSTER>(s, gen)) return;
                const int64_t slots = a.nr * s.lanes[side];
                for (int64_t t0 = (int64_t)blockIdx.x * kThreads; t0 < slots;
                     t0 += (int64_t)gridDim.x * kThreads)
                    merge_slot(t0 + tid, a.partial, a.splits, a.nr, a.rnorm, a.rlogw2, a.eps_ln2,
                               a.pot, a.rows + D, fma_stride(D), ref ? a.fix_list : nullptr,
                               ref ? a.fix_count : nullptr, s.lanes[side]);
            }
            if (!phase_barrier<CLUSTER>(s, gen)) return;
            if (ref) {
                // the other side's list was read completely before this point
                if (blockIdx.x == 0 && tid == 0) {
                    const HalfArgs& o = s.h[side ^ 1];
                    const unsigned int oc = min(o.fix_count[0], (unsigned int)o.nr);
                    if (o.fix_stats != nullptr && it - (side == 0 ? 1 : 0) >= s.ref_from) {
                        o.fix_stats[0] += 1ull;
                        o.fix_stats[1] += oc;
                    }
                    o.fix_count[0] = 0u;
                }
                const unsigned int cnt =
                    min(*(volatile unsigned int*)&a.fix_count[0], (unsigned int)a.nr);
                if (cnt > 0) {   // every block read the same count (the list is complete)
                    const unsigned int warps = gridDim.x * (kThreads / 32);
                    for (unsigned int w = blockIdx.x * (kThreads / 32) + (tid >> 5); w < cnt;
                         w += warps) {
                        const int64_t row = a.fix_list[w];
                        if (!FS_IDX_OK(row, a.nr, 4)) continue;
                        fix_row<D>(a, row, lane);
                    }
                    if (!phase_barrier<CLUSTER>(s, gen)) return;
                }
            }
        }
    }
    // the last half's list: counted and reset by block 0 after the final barrier
    if (blockIdx.x == 0 && tid == 0 && s.n_iter > s.ref_from) {
        const HalfArgs& o = s.h[1];
        if (o.fix_stats != nullptr) {
            o.fix_stats[0] += 1ull;
            o.fix_stats[1] += min(o.fix_count[0], (unsigned int)o.nr);
        }
        o.fix_count[0] = 0u;
    }
}

// One block arrives, the other never does (a wait that must run out).
__global__ void k_barrier_selftest(unsigned int* bar, uint32_t* err, uint64_t timeout_ns) {
    if (blockIdx.x != 0) return;
    unsigned int gen = 0;
    grid_barrier(bar, gen, err, timeout_ns);
}

template <int D>
int solve_small_blocks_t() {
    static std::atomic<int> cached{0};
    int v = cached.load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k_solve_small<D, fma_row_pairs(D), false>,
                                                          kThreads, 0) != cudaSuccess || v < 1)
            v = 1;
        cached.store(v, std::memory_order_relaxed);
    }
    return v;
}

constexpr int kClusterSolveMax = 16;   // blocks of a one-cluster solve (non-portable above 8)

// Largest one-cluster grid the device schedules for the solve kernel (0: none).
template <int D>
int cluster_solve_max_t() {
    static std::atomic<int> cached{-1};
    int v = cached.load(std::memory_order_relaxed);
    if (v < 0) {
        v = 0;
        const void* fn = (const void*)k_solve_small<D, fma_row_pairs(D), true>;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            (void)cudaGetLastError();
        for (int c = kClusterSolveMax; c >= 2 && v == 0; c /= 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)c);
            cfg.blockDim = dim3(kThreads);
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = (unsigned)c;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) == cudaSuccess && clusters >= 1) v = c;
            else (void)cudaGetLastError();
        }
        cached.store(v, std::memory_order_relaxed);
    }
    return v;
}

template <int D>
cudaError_t launch_solve_small_t(const SmallArgs& a, int sms, cudaStream_t s) {
    // no more blocks than work items of the larger half-update: every block
    // takes part in every barrier
    const int64_t items = std::max(a.row_blocks[0] * a.h[0].splits, a.row_blocks[1] * a.h[1].splits);
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(items, (int64_t)solve_small_blocks_t<D>() * sms));
    SmallArgs args = a;
    cudaError_t e;
    if (blocks <= cluster_solve_max_t<D>()) {
        // the whole grid as one cluster: the same blocks and work items, the
        // hardware cluster barrier between phases
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(kThreads);
        cfg.stream = s;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)blocks;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, k_solve_small<D, fma_row_pairs(D), true>, args);
    } else {
        void* params[] = {&args};
        e = cudaLaunchCooperativeKernel((const void*)k_solve_small<D, fma_row_pairs(D), false>,
                                        dim3((unsigned)blocks), dim3(kThreads), params, 0, s);
    }
    count_launch();
    return e;
}

// ---------------------------------------------------------------------------
// Plan application (Method 3): out_i = sum_j P_ij V_j with
//   P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps) = a_i 2^{phi_i} 2^{s_ij},
// phi_i = (f_i - |x~_i|^2) L/eps and s_ij the f-update score built from g.
// Each thread owns one row and KC columns of V; a running max M keeps the
// accumulator O = sum_j 2^{s_ij - M} V_j in range, so out_i = a_i 2^{phi_i+M} O.

constexpr int kApplyThreads = 128;
constexpr int kApplyChunk = 256;

template <int D, int KC, bool TAN>
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
    // APPLY_TAN: t_ij = u_i . (y~_j - x~_i) = u_i . y~_j - c_i (the centring cancels)
    float u[D];
    float ci = 0.f, sig = 0.f;
    if (TAN) {
#pragma unroll
        for (int k = 0; k < D; ++k) {
            u[k] = k < a.d ? a.U[rr * a.d + k] : 0.f;
            ci = fmaf(u[k], a.rows[rr * DS + k], ci);
        }
    }
    float M = -INFINITY;
    float O[KC];
#pragma unroll
    for (int c = 0; c < KC; ++c) O[c] = 0.f;

    for (int64_t cb = c0; cb < c1; cb += kApplyChunk) {
        const int ncol = (int)min((int64_t)kApplyChunk, c1 - cb);
        __syncthreads();
        const float4* src = reinterpret_cast<const float4*>(a.cols + cb * DS);
        for (int e = tid; e < ncol * (DS / 4); e += kApplyThreads)
            if (FS_IDX_OK(cb * (DS / 4) + e, a.m * (DS / 4), 5)) sc[e] = src[e];
        for (int e = tid; e < ncol * KC; e += kApplyThreads) {
            const int j = e / KC, c = e - j * KC;
            const int64_t vi = (cb + j) * a.k + kc0 + c;
            sv[e] = c < kw && FS_IDX_OK(vi, a.m * (int64_t)a.k, 6) ? a.V[vi] : 0.f;
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
                if (TAN) sig *= r;
                M = sij;
            }
            float p = ex2(sij - M);
            if (TAN) {
                float t = -ci;
#pragma unroll
                for (int k = 0; k < D; ++k) t = fmaf(u[k], cv[k], t);
                p *= t;
                sig += p;
            }
#pragma unroll
            for (int c = 0; c < KC; ++c) O[c] = fmaf(p, sv[j * KC + c], O[c]);
        }
    }
    if (row >= a.n) return;
    const int pk_stride = a.k + 1 + (TAN ? 1 : 0);
    if (a.splits > 1) {
        const int64_t base = ((int64_t)blockIdx.y * a.n + row) * pk_stride;
        [[maybe_unused]] const int64_t plen = (int64_t)a.splits * a.n * pk_stride;   // index checks
        if (blockIdx.z == 0 && FS_IDX_OK(base, plen, 7)) a.partial[base] = M;
        if (TAN && blockIdx.z == 0 && FS_IDX_OK(base + 1 + a.k, plen, 7)) a.partial[base + 1 + a.k] = sig;
        for (int c = 0; c < kw; ++c)
            if (FS_IDX_OK(base + 1 + kc0 + c, plen, 7)) a.partial[base + 1 + kc0 + c] = O[c];
        return;
    }
    const float w = exp2f(a.phi[row] + M);
    if (TAN && blockIdx.z == 0) a.out2[row] = a.a[row] * (w * sig);
    for (int c = 0; c < kw; ++c) {
        const float t = w * O[c];
        float o;
        if (a.mode == APPLY_PV || a.mode == APPLY_TAN) o = a.a[row] * t;
        else if (a.mode == APPLY_BARY) o = t;
        else o = 2.f * a.a[row] * (a.X[row * a.d + kc0 + c] - t);
        if (FS_IDX_OK(row * a.k + kc0 + c, a.n * (int64_t)a.k, 8)) a.out[row * a.k + kc0 + c] = o;
    }
}

template <int D>
cudaError_t launch_apply_fma_t(const ApplyArgs& a, cudaStream_t s) {
    const unsigned kchunks16 = (unsigned)((a.k + 15) / 16);
    dim3 grid((unsigned)((a.n + kApplyThreads - 1) / kApplyThreads), (unsigned)a.splits);
    const bool tan = a.mode == APPLY_TAN;
    if (a.k <= 4) {
        grid.z = 1;
        if (tan) k_apply_fma<D, 4, true><<<grid, kApplyThreads, 0, s>>>(a);
        else k_apply_fma<D, 4, false><<<grid, kApplyThreads, 0, s>>>(a);
    } else {
        grid.z = kchunks16;
        if (tan) k_apply_fma<D, 16, true><<<grid, kApplyThreads, 0, s>>>(a);
        else k_apply_fma<D, 16, false><<<grid, kApplyThreads, 0, s>>>(a);
    }
    count_launch();
    return cudaGetLastError();
}

__global__ void k_merge_apply(ApplyArgs a) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.n) return;
    const int pk_stride = a.k + 1 + (a.mode == APPLY_TAN ? 1 : 0);
    const int64_t stride = (int64_t)a.n * pk_stride;
    float M = -INFINITY;
    for (int sp = 0; sp < a.splits; ++sp) M = fmaxf(M, a.partial[sp * stride + i * pk_stride]);
    const float w = exp2f(a.phi[i] + M);
    if (a.mode == APPLY_TAN) {
        float sig = 0.f;
        for (int sp = 0; sp < a.splits; ++sp) {
            const float* p = a.partial + sp * stride + i * pk_stride;
            sig += p[1 + a.k] * ex2(p[0] - M);
        }
        a.out2[i] = a.a[i] * (w * sig);
    }
    for (int c = 0; c < a.k; ++c) {
        float O = 0.f;
        for (int sp = 0; sp < a.splits; ++sp) {
            const float* p = a.partial + sp * stride + i * pk_stride;
            O += p[1 + c] * ex2(p[0] - M);
        }
        const float t = w * O;
        float o;
        if (a.mode == APPLY_PV || a.mode == APPLY_TAN) o = a.a[i] * t;
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

namespace {
template <int D, int MODE>
int half_fma_residency() {
    static std::atomic<int> cached{0};
    int v = cached.load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k_half_fma<D, fma_row_pairs(D), MODE>,
                                                          kThreads, 0) != cudaSuccess || v < 1)
            v = 1;
        cached.store(v, std::memory_order_relaxed);
    }
    return v;
}
}  // namespace

int fma_half_blocks_per_sm(int D, bool folded) {
    if (folded) {
        switch (D) {
            case 2: return half_fma_residency<2, 2>();
            case 3: return half_fma_residency<3, 2>();
            case 4: return half_fma_residency<4, 2>();
            default: break;
        }
    }
    switch (D) {
        case 2: return half_fma_residency<2, 1>();
        case 3: return half_fma_residency<3, 1>();
        case 4: return half_fma_residency<4, 1>();
        case 8: return half_fma_residency<8, 1>();
        default: return half_fma_residency<16, 1>();
    }
}

cudaError_t launch_barrier_selftest(unsigned int* bar, uint32_t* err, uint64_t timeout_ns,
                                    cudaStream_t s) {
    void* params[] = {&bar, &err, &timeout_ns};
    const cudaError_t e = cudaLaunchCooperativeKernel((const void*)k_barrier_selftest, dim3(2),
                                                      dim3(32), params, 0, s);
    count_launch();
    return e;
}

// Lanes per row of the split merge: each lane folds up to kMergePerLane of
// the row's partials in split order, then the lanes combine in a butterfly.
// Few lanes keep the one-launch solve's merge phase to one pass over its
// threads: 45 splits of 10^4 rows merge in 3.7 us with 8 lanes, 6.1 us with
// 32 (a lane per split up to 32) and 31.3 against 29.9 us per half-update
// with 4 (twelve partials a lane).
constexpr int kMergePerLane = 6;
int merge_lanes(int splits) {
    int lanes = 1;
    while (lanes * kMergePerLane < splits && lanes < 32) lanes *= 2;
    return lanes;
}

cudaError_t launch_solve_small(int D, const SmallArgs& a, int sms, cudaStream_t s) {
    switch (D) {
        case 2: return launch_solve_small_t<2>(a, sms, s);
        case 3: return launch_solve_small_t<3>(a, sms, s);
        case 4: return launch_solve_small_t<4>(a, sms, s);
        case 8: return launch_solve_small_t<8>(a, sms, s);
        case 16: return launch_solve_small_t<16>(a, sms, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge_lse(const float2* partial, int splits, int64_t nr, const float* rnorm,
                             const float* rlogw2, float eps_ln2, float* pot, float* bias,
                             int64_t bias_stride, cudaStream_t s, int* fix_list,
                             unsigned int* fix_count) {
    const int lanes = merge_lanes(splits);
    const int64_t threads = nr * lanes;
    k_merge_lse<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
        partial, splits, nr, rnorm, rlogw2, eps_ln2, pot, bias, bias_stride, fix_list, fix_count,
        lanes);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_fix_fma(int D, const HalfArgs& a, cudaStream_t s) {
    switch (D) {
        case 2: return launch_fix_fma_t<2>(a, s);
        case 3: return launch_fix_fma_t<3>(a, s);
        case 4: return launch_fix_fma_t<4>(a, s);
        case 8: return launch_fix_fma_t<8>(a, s);
        case 16: return launch_fix_fma_t<16>(a, s);
        default: return cudaErrorInvalidValue;
    }
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

FS_BOUNDS_READER(bounds_take_fma)

cudaError_t launch_merge_apply(const ApplyArgs& a, cudaStream_t s) {
    k_merge_apply<<<(unsigned)((a.n + 127) / 128), 128, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs

// Internal declarations shared by the translation units of libflashsinkhorn.
//
// Notation (base-2 folded form of the pages' Proposition 1).  With centred
// points x~ = x - t, y~ = y - t (t is any common shift; the cost is invariant),
// L = log2(e) and kappa = 2 L / eps, the f-update of the pages,
//     f_i = -eps LSE_j[(g_j - C_ij)/eps + log b_j],
// becomes
//     s_ij  = kappa x~_i . y~_j + beta_j,    beta_j = (g_j - |y~_j|^2) L/eps + log2 b_j
//     f_i   = |x~_i|^2 - eps ln2 * log2 sum_j 2^{s_ij}
// and the bias the following g-update needs is
//     alpha_i = (f_i - |x~_i|^2) L/eps + log2 a_i = log2 a_i - log2 sum_j 2^{s_ij}.
// The g-update is the same computation with the roles of (X, a, f, alpha) and
// (Y, b, g, beta) exchanged.  beta and alpha are the pages' g_hat + delta and
// f_hat + gamma, divided by eps and written in base 2.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>

namespace fs {

constexpr double kLog2e = 1.4426950408889634074;   // log2(e)
constexpr double kLn2 = 0.69314718055994530942;    // ln(2)

// Kernel launches issued by the library (reported by fs_launch_count).
extern std::atomic<int64_t> g_launches;
inline void count_launch(int64_t k = 1) { g_launches.fetch_add(k, std::memory_order_relaxed); }

// Device error word bits (set by bounded waits; read by fs_check).
enum : uint32_t {
    ERR_TIMEOUT_PRODUCER = 1u,
    ERR_TIMEOUT_MMA = 2u,
    ERR_TIMEOUT_EPILOGUE = 4u,
    ERR_TIMEOUT_BARRIER = 16u    // a grid barrier of the one-launch solve gave up
};

// ---------------------------------------------------------------------------
// device helpers

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// packed fp32 arithmetic: two lanes per instruction (sm_100 family)
__device__ __forceinline__ uint64_t pk(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ void upk(uint64_t r, float& x, float& y) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ---------------------------------------------------------------------------
// FMA path: packed operand arrays.  Row r of a packed array holds the centred
// coordinates of a point, zero-padded to D, then its current bias (alpha or
// beta) at index D, padded to a stride DS that is a multiple of 4 floats.

__host__ __device__ constexpr int fma_pad_dim(int d) { return d <= 2 ? 2 : d <= 3 ? 3 : d <= 4 ? 4 : d <= 8 ? 8 : 16; }
__host__ __device__ constexpr int fma_stride(int D) { return ((D + 1) + 3) / 4 * 4; }
constexpr int kFmaMaxDim = 16;
// Half-update rows per thread come in pairs (packed f32x2 lanes); blocks are
// 256 threads, so a block covers 512 * fma_row_pairs(D) rows.
__host__ __device__ constexpr int fma_row_pairs(int D) { return D <= 4 ? 2 : 1; }
constexpr int64_t fma_rows_per_block(int D) { return 512 * fma_row_pairs(D); }

// Half-update on the FMA path.  rows: packed array of the side being
// updated (nr rows); cols: packed array of the other side (nc rows) whose
// bias slot holds beta (or alpha).  Writes pot[i] and the row bias into
// rows[i*DS + D] (splits == 1), or (max, sum) partials (splits > 1).
struct HalfArgs {
    float* rows;            // packed [nr x DS]; bias slot written
    const float* cols;      // packed [nc x DS]
    int64_t nr, nc;
    float kappa;            // 2 log2(e) / eps
    float eps_ln2;          // eps * ln 2
    const float* rnorm;     // |x~_i|^2 [nr]
    const float* rlogw2;    // log2 of the row weights [nr]
    float* pot;             // potential out [nr]
    float2* partial;        // [splits x nr] or nullptr
    int splits;
    int64_t cols_per_split;
    // Reference offsets: with use_ref set, each row's exponent offset is the
    // LSE of its previous half-update (log2 w_i minus its bias slot) instead
    // of an online max; rows whose sum leaves the guarded range are appended
    // to fix_list (fix_count[0] entries) for launch_fix_fma.
    int use_ref;              // 0 online max, 1 reference offsets, 2 reference offsets
                              // folded per CTA (rows in Morton order; d <= 4)
    int* fix_list;            // [nr]
    unsigned int* fix_count;  // [2], zero before the first guarded half-update
    // Cumulative fixup statistics [2] (fixup launches, rows recomputed), or
    // nullptr; the fixup kernel's last block adds to them.
    unsigned long long* fix_stats;
};
cudaError_t launch_half_fma(int D, const HalfArgs& a, cudaStream_t s);

// The whole solve as one cooperative launch (small problems): n_iter
// iterations of (f-half, g-half), each half-update's work items, split merge
// and fixups separated by bounded grid barriers.  h[0] / h[1] are the two
// halves' arguments as for launch_half_fma (with their own fixup lists).
struct SmallArgs {
    HalfArgs h[2];
    int64_t row_blocks[2];
    int lanes[2];             // merge lanes per row (as launch_merge_lse chooses)
    int n_iter;
    int ref_from;             // first iteration with reference offsets (n_iter: none)
    unsigned int* bar;        // [2] grid barrier (arrivals, generation), zero before first use
    uint32_t* err;            // device error word
    uint64_t timeout_ns;      // a barrier wait gives up after this long
};
cudaError_t launch_solve_small(int D, const SmallArgs& a, int sms, cudaStream_t s);
// Failure-detection self-test of that grid barrier: two co-resident blocks,
// one of which never arrives; the other's wait gives up after timeout_ns and
// sets ERR_TIMEOUT_BARRIER.  bar: [2] zeroed device words.
cudaError_t launch_barrier_selftest(unsigned int* bar, uint32_t* err, uint64_t timeout_ns,
                                    cudaStream_t s);
// lanes per row of the split merge for `splits` partials
int merge_lanes(int splits);
// Recompute the listed rows with the online max; resets the list.
cudaError_t launch_fix_fma(int D, const HalfArgs& a, cudaStream_t s);
// Blocks of the half-update kernel for padded dimension D resident per SM
// (folded: the kernel of the folded-offset mode, d <= 4).
int fma_half_blocks_per_sm(int D, bool folded = false);

// Merge of split partials: LSE2 = M + log2 sum_s S_s 2^{M_s - M} in split
// order, then pot = rnorm - eps ln2 LSE2 and bias = rlogw2 - LSE2.
// With fix_list set, rows whose merged sum leaves the guarded range of a
// reference-offset half-update are appended to it.
cudaError_t launch_merge_lse(const float2* partial, int splits, int64_t nr, const float* rnorm,
                             const float* rlogw2, float eps_ln2, float* pot, float* bias,
                             int64_t bias_stride, cudaStream_t s, int* fix_list = nullptr,
                             unsigned int* fix_count = nullptr);

// Plan application on the FMA path.
// APPLY_TAN weights each plan entry by t_ij = u_i . (y_j - x_i) for row
// directions U (n x d): out_i = sum_j P_ij t_ij V_j and out2_i = sum_j P_ij t_ij
// (the plan's tangent along X + tU at fixed potentials, up to -2/eps).
enum ApplyMode : int { APPLY_PV = 0, APPLY_BARY = 1, APPLY_GRAD = 2, APPLY_TAN = 3 };
struct ApplyArgs {
    const float* rows;      // packed [n x DS] (centred x~)
    const float* cols;      // packed [m x DS] with beta from the given g
    const float* phi;       // (f_i - |x~_i|^2) L/eps  [n]
    const float* V;         // [m x k]
    int k;
    int64_t n, m;
    float kappa;
    const float* a;         // weights [n]
    const float* X;         // raw X [n x d] (grad mode)
    int d;
    float* out;             // [n x k]
    float* partial;         // [splits x n x (k+1)] ([.. x (k+2)] in APPLY_TAN) or nullptr
    int splits;
    int64_t cols_per_split;
    int mode;
    const float* U;         // APPLY_TAN: row directions [n x d]
    float* out2;            // APPLY_TAN: sum_j P_ij t_ij [n]
};
cudaError_t launch_apply_fma(int D, const ApplyArgs& a, cudaStream_t s);
cudaError_t launch_merge_apply(const ApplyArgs& a, cudaStream_t s);

// ---------------------------------------------------------------------------
// Preparation kernels.

// Per-dimension sums of the rows of X and Y in double, in a fixed order:
// partial[blk * d + k] over row blocks, then shift[k] = total / (n + m).
cudaError_t launch_shift(const float* X, int64_t n, const float* Y, int64_t m, int d,
                         double* partial, int nblk_max, float* shift, cudaStream_t s);

// FMA path: centre, pack, norms and log2-weights of one side.  If `pot` is
// non-null the bias slot is filled from it: bias = (pot - |p~|^2) L/eps + log2 w.
// With `perm`, packed row i is the caller's row perm[i] (P, w and pot are read
// there); outputs are in the permuted order.
cudaError_t launch_pack_fma(const float* P, const float* w, const float* pot, int64_t rows, int d,
                            int D, const float* shift, float l_over_eps, float* packed,
                            float* norm, float* logw2, cudaStream_t s, const int* perm = nullptr);

// dst[perm[i]] = src[i], i < rows (back from a permuted order).
cudaError_t launch_scatter_rows(const float* src, const int* perm, int64_t rows, float* dst,
                                cudaStream_t s);

// phi_i = (f_i - |x~_i|^2) L/eps (apply).
cudaError_t launch_phi(const float* f, const float* norm, int64_t n, float l_over_eps, float* phi,
                       cudaStream_t s);

// Count NaN/Inf in v (atomic counter, integer).
cudaError_t launch_count_nonfinite(const float* v, int64_t len, unsigned int* counter,
                                   cudaStream_t s);

}  // namespace fs

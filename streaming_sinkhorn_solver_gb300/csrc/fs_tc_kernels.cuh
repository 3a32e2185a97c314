// Launch interfaces of the tensor-core path (kernels in fs_tc.cu / fs_tc_apply.cu).
#pragma once

#include "fs_internal.cuh"

namespace fs {
namespace tc {

constexpr int BM = 128;                 // rows of a tile (TMEM lanes)
constexpr int BK = 64;                  // fp16 elements per 128-byte swizzled row
constexpr int CHUNK_BYTES = BM * BK * 2;  // one 128 x 64 fp16 chunk = 16 KB
constexpr int BN = 128;                 // columns of a score tile (TMEM columns per buffer)
constexpr int kEpiWarps = 4;            // warps of one epilogue group (one thread per tile row)
// half-update kernel
constexpr int kHalfGroups = 2;          // epilogue groups, alternating score tiles
constexpr int kTmemBufs = 4;            // score tiles in flight in TMEM (tile t -> t mod 4)
constexpr int kHalfThreads = 32 * (2 + kHalfGroups * kEpiWarps);
constexpr int kTmemCols = kTmemBufs * BN;
constexpr int kMaxStages = 8;           // shared-memory ring depth is set by the free space
constexpr int kSmemLimit = 232448;      // dynamic shared memory per block on sm_103
constexpr int kMaxResidentChunks = 8;   // Q stays in shared memory up to d = 512

// Operand tiles: a cloud of `rows` points becomes ceil(rows/128) tiles of
// nch = ceil(d/64) chunks, each chunk 128 rows x 64 fp16 (16 KB) in the
// K-major 128-byte-swizzled order; padding rows and dimensions are zero.
struct TcHalfArgs {
    const void* Q;          // row-side tiles
    const void* K;          // column-side tiles
    const float* cbias;     // column bias, col_tiles*128 entries, padding = -inf
    const float* kscale;    // device scalar: kappa 2^-(ex+ey)
    int64_t nr, nc;
    int nch;
    int col_tiles;
    int tiles_per_split;
    int splits;
    int stages;             // ring depth (from half_stages)
    int raster_pairs;       // CTA-pair kernel: pairs per launch-order group (0 = all)
    float eps_ln2;
    const float* rnorm;     // |x~|^2 of the rows; nullptr = write log2-sum-exp only
    const float* rlogw2;    // log2 of the row weights
    float* pot;             // potential (or log2-sum-exp) of each row
    float* rbias;           // bias of the rows for the next half-update
    float2* partial;        // (max, sum) per split and row when splits > 1
    uint32_t* err;          // device error word
    // Reference offsets: with use_ref set, a row's exponent
    // offset is its previous LSE, rlogw2 - rbias, instead of a running max;
    // rows whose sum leaves the guarded range go to fix_list for
    // launch_fix_tc.
    int use_ref;
    int* fix_list;            // [nr]
    unsigned int* fix_count;  // [2], zero before the first guarded half-update
};

// Groups of the reference-offset half-update (fs_tc_ref.cu): four groups of
// four warps, one per TMEM buffer, each issuing its own copies and MMAs.
constexpr int kRefGroups = 4;
// Epilogue groups of the CTA-pair half-update with reference offsets: two
// per TMEM buffer, each owning half of its columns (one group per buffer,
// with the registers of 10 warps instead of 18, ran 2 % slower at d = 512).
constexpr int kPairRefGroups = 4;
// Threads of the CTA-pair half-update: producer, MMA warp and the epilogue
// groups (two with online maxima).
constexpr int half_threads(bool ref) {
    return 32 * (2 + (ref ? kPairRefGroups : kHalfGroups) * kEpiWarps);
}

// Guarded range of a reference-offset sum (see the FMA path).
constexpr float kTcMinRefSum = 5.421010862427522e-20f;   // 2^-64
constexpr float kTcMaxRefSum = 8.507059173023462e+37f;   // 2^126

// FP32 recomputation of the rows a guarded half-update listed: one warp per
// row over all columns, centred coordinates, online max.
struct TcFixArgs {
    const float* R;           // raw coordinates of the updated side [nr x d]
    const float* C;           // raw coordinates of the other side [nc x d]
    const float* shift;       // [d]
    int d;
    float kappa;              // 2 log2(e) / eps
    const float* cbias;       // column bias [nc] (beta or alpha)
    int64_t nr, nc;
    float eps_ln2;
    const float* rnorm;
    const float* rlogw2;
    float* pot;
    float* rbias;
    int* fix_list;
    unsigned int* fix_count;
    unsigned long long* fix_stats;   // [2] launches, rows recomputed (or nullptr)
};
constexpr int kFixMaxDim = 1024;   // reference offsets on the tensor path up to this d
cudaError_t launch_fix_tc(const TcFixArgs& a, cudaStream_t s);

cudaError_t launch_prep_side(const float* P, const float* w, int64_t rows, int d,
                             const float* shift, float* norm, float* logw2,
                             unsigned int* absmax_bits, cudaStream_t s);
cudaError_t launch_scales(const unsigned int* absmax_bits, float kappa, float* params,
                          cudaStream_t s);
cudaError_t launch_to_tiles(const float* P, int64_t rows, int d, const float* shift,
                            const float* scale_ptr, int nch, int64_t row_tiles, void* out,
                            void* out_lo, cudaStream_t s);
cudaError_t launch_bias_init(const float* pot, const float* norm, const float* logw2,
                             float l_over_eps, int64_t rows, int64_t rows_pad, float* bias,
                             cudaStream_t s);
// An opaque 128-byte TMA descriptor (CUtensorMap), passed by value to kernels.
struct alignas(64) TensorMap128 {
    unsigned char bytes[128];
};

// CTA-pair variant (fs_tc_pair.cu): M = 256 over two CTAs, 256-column tiles
// (col_tiles / tiles_per_split count 256-column tiles; row_tiles even; K has
// an even number of 128-row tiles and the bias 256 entries per tile).  tmQ /
// tmK are chunk maps (make_chunk_tmap) over a.Q / a.K.
int pair_stages(int nch, bool qres);
size_t pair_smem_bytes(int nch, bool qres, int stages);
cudaError_t launch_half_pair(const TcHalfArgs& a, const TensorMap128& tmQ,
                             const TensorMap128& tmK, int row_tiles, bool qres, cudaStream_t s);

int half_stages(int nch, bool qres);    // deepest ring that fits next to resident Q
size_t half_smem_bytes(int nch, bool qres, int stages);
// online-max kernel, or with a.use_ref set the reference-offset kernel
// (requires qres and nch <= 2)
cudaError_t launch_half_tc(const TcHalfArgs& a, int row_tiles, bool qres, cudaStream_t s);
cudaError_t launch_half_ref(const TcHalfArgs& a, int row_tiles, cudaStream_t s);

// ---------------------------------------------------------------------------
// Plan application.  Values V (m x k) are stored transposed per column tile:
// tile j holds, for each of its two 64-point halves kq, kpad rows (one per
// output column n) of 64 fp16 values in the K-major 128-byte-swizzled order,
// i.e. byte ((j*2 + kq)*kpad + n)*128 + swizzled offset of point p.
constexpr int kApplyStages = 2;         // (K hi, K lo, Q hi, Q lo) chunk sets in flight
// Output columns per CTA (TMEM columns of O): 256 when the scores of a tile
// take long enough (d >= 256) to hide the load of the next value tile into a
// single 64 KB slot, else 128 with two value slots.  Every 256 columns of
// output recompute the scores once.
__host__ __device__ constexpr int apply_kv(int nch, int kpad) { return nch >= 4 && kpad > 128 ? 256 : 128; }
constexpr int kApplyThreads = 32 * (2 + kEpiWarps);   // producer, MMA, one epilogue group
constexpr int kApplyTmemCols = 512;     // 2 score buffers + O, rounded to a power of two

// Scores are formed in split precision, S = Qh Kh^T + Qh Kl^T + Ql Kh^T with
// hi = fp16(v) and lo = fp16(v - hi): an error near 2^-22 instead of 2^-11,
// because a plan entry carries the score's absolute error as a relative one.
struct TcApplyArgs {
    const void* Q;          // row-side tiles (hi part)
    const void* K;          // column-side tiles (hi part)
    const void* Qlo;        // row-side remainders
    const void* Klo;        // column-side remainders
    const void* VT;         // transposed value tiles
    const float* cbias;     // beta built from g, padding -inf
    const float* kscale;    // device scalar: kappa 2^-(ex+ey)
    const float* lse2;      // log2 sum_j 2^{s_ij} per row (pre-pass)
    const float* phi;       // (f_i - |x~_i|^2) L/eps per row
    const float* vinv;      // device scalar: 1 / (power-of-two scale of V)
    const float* shift;     // centring shift (barycentric / gradient modes)
    const float* a;         // row weights
    const float* X;         // raw rows (gradient mode), n x d
    int64_t nr, nc;
    int nch, col_tiles, tiles_per_split, splits;
    int k, kpad;
    int mode;               // APPLY_PV / APPLY_BARY / APPLY_GRAD / APPLY_TAN
    float* out;             // n x k
    float* partial;         // splits x n x (k+1): unscaled sums, then sum_j p_ij
    uint32_t* err;
    // APPLY_TAN: each p_ij is weighted by t_ij = u_i . (y_j - x_i), formed on
    // the tensor cores as U K^T (split precision, a second TMEM buffer) minus
    // the row constant u_i . x~_i; out2_i = a_i W_i sum_j p_ij t_ij.
    const void* U;          // row-direction tiles (hi), same layout as Q
    const void* Ulo;        // row-direction remainders
    const float* tparams;   // [0] scale of U K^T to t 2^et, [1] 2^et, [2] 2^-et
    const float* crow;      // u_i . x~_i per row
    float* out2;            // n
};

size_t apply_smem_bytes();
cudaError_t launch_apply_tc(const TcApplyArgs& a, int row_tiles, cudaStream_t s);
cudaError_t launch_merge_apply_tc(const TcApplyArgs& a, cudaStream_t s);
// transposed value tiles from V (m x k, row-major); shift subtracted if given
cudaError_t launch_vt_tiles(const float* V, int64_t m, int k, int kpad, const float* shift,
                            const float* scale_ptr, int64_t col_tiles, void* out,
                            cudaStream_t s);
// tangent application: crow_i = u_i . x~_i and maxima of |u_i|^2, |u_ik| into
// bits[0..1]; then the scales of the tangent weights from bits[0..3] (bits[2..3]:
// max |x~_i|^2, max |y~_j|^2) and the column cloud's tile scale
cudaError_t launch_tan_rows(const float* U, const float* X, int64_t rows, int d, const float* shift,
                            float* crow, unsigned int* bits, cudaStream_t s);
cudaError_t launch_tan_params(const unsigned int* bits, const float* yscale, float* tparams,
                              cudaStream_t s);
// max |V| as ordered float bits (atomicMax)
cudaError_t launch_absmax(const float* V, int64_t len, unsigned int* bits, cudaStream_t s);
// params[0] = 2^e with max|V| 2^e in [2^14, 2^15), params[1] = 2^-e
cudaError_t launch_value_scale(const unsigned int* bits, float* params, cudaStream_t s);

}  // namespace tc
}  // namespace fs

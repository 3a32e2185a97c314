// Launch interfaces of the tensor-core path (kernels in fs_tc.cu / fs_tc_apply.cu).
#pragma once

#include "fs_internal.cuh"

namespace fs {
namespace tc {

constexpr int BM = 128;                 // rows of a tile (TMEM lanes)
constexpr int BK = 64;                  // fp16 elements per 128-byte swizzled row
constexpr int CHUNK_BYTES = BM * BK * 2;  // one 128 x 64 fp16 chunk = 16 KB
constexpr int BN = 128;                 // columns of a score tile (TMEM columns per buffer)
constexpr int kStages = 4;              // shared-memory ring depth (chunks)
constexpr int kTmemBufs = 2;            // score tiles in flight in TMEM
constexpr int kEpiWarps = 4;            // epilogue warps (one thread per tile row)
constexpr int kHalfThreads = 32 * (2 + kEpiWarps);
constexpr int kTmemCols = kTmemBufs * BN;
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
    float eps_ln2;
    const float* rnorm;     // |x~|^2 of the rows; nullptr = write log2-sum-exp only
    const float* rlogw2;    // log2 of the row weights
    float* pot;             // potential (or log2-sum-exp) of each row
    float* rbias;           // bias of the rows for the next half-update
    float2* partial;        // (max, sum) per split and row when splits > 1
    uint32_t* err;          // device error word
};

cudaError_t launch_prep_side(const float* P, const float* w, int64_t rows, int d,
                             const float* shift, float* norm, float* logw2,
                             unsigned int* absmax_bits, cudaStream_t s);
cudaError_t launch_scales(const unsigned int* absmax_bits, float kappa, float* params,
                          cudaStream_t s);
cudaError_t launch_to_tiles(const float* P, int64_t rows, int d, const float* shift,
                            const float* scale_ptr, int nch, int64_t row_tiles, void* out,
                            cudaStream_t s);
cudaError_t launch_bias_init(const float* pot, const float* norm, const float* logw2,
                             float l_over_eps, int64_t rows, int64_t rows_pad, float* bias,
                             cudaStream_t s);
size_t half_smem_bytes(int nch, bool qres);
cudaError_t launch_half_tc(const TcHalfArgs& a, int row_tiles, bool qres, cudaStream_t s);

}  // namespace tc
}  // namespace fs

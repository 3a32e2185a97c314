// Bounds checks of global-memory indices for debug builds.
//
// Built with -DFS_DEBUG_BOUNDS (build(debug_bounds=True), which writes
// libflashsinkhorn_dbg.so), every checked access tests its index against the
// size of its buffer; an index outside records the first violation of its
// translation unit, (site << 48) | (index & 0xffffffffffff), in a device
// word and the access is skipped, so a bad index is reported instead of
// faulting.  fs_debug_bounds() reads and clears the words of every
// instrumented translation unit.  In release builds FS_IDX_OK is the
// constant true and nothing is compiled.
//
// Site codes: 1-19 fs_fma.cu, 20-29 fs_prep.cu, 30-59 fs_sparse.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fs {

#ifdef FS_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
// one word per translation unit that includes this header
static __device__ unsigned long long g_bounds_word;

__device__ __forceinline__ bool idx_ok(int64_t i, int64_t n, unsigned int site) {
    if (i >= 0 && i < n) return true;
    atomicCAS(&g_bounds_word, 0ull,
              ((unsigned long long)site << 48) | ((unsigned long long)i & 0xffffffffffffull));
    return false;
}
#define FS_IDX_OK(i, n, site) ::fs::idx_ok((int64_t)(i), (int64_t)(n), (site))
#define FS_BOUNDS_READER(NAME)                                                          \
    cudaError_t NAME(unsigned long long* out) {                                         \
        cudaError_t e = cudaMemcpyFromSymbol(out, g_bounds_word, sizeof(*out));         \
        if (e != cudaSuccess) return e;                                                 \
        const unsigned long long zero = 0;                                              \
        return cudaMemcpyToSymbol(g_bounds_word, &zero, sizeof(zero));                  \
    }
#else
constexpr bool kDebugBounds = false;
#define FS_IDX_OK(i, n, site) true
#define FS_BOUNDS_READER(NAME)                  \
    cudaError_t NAME(unsigned long long* out) { \
        *out = 0;                               \
        return cudaSuccess;                     \
    }
#endif

// Readers of the instrumented translation units (read and clear).
cudaError_t bounds_take_fma(unsigned long long* out);
cudaError_t bounds_take_prep(unsigned long long* out);
cudaError_t bounds_take_sparse(unsigned long long* out);

}  // namespace fs

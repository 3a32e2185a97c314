// Morton (Z-order) permutation of two low-dimensional clouds, shared by the
// block-sparse solver and the dense FMA path.
//
// Both clouds are quantised on one joint bounding box (2^B cells per axis,
// B = min(21, floor(63 / d)): the interleaved code fits 64 bits) and sorted
// by their interleaved codes with a stable radix sort, so equal codes keep
// the caller's order.  Consecutive points of the result form
// compact groups in space ("FlashSinkhorn 2: Block-Sparse Entropic Optimal
// Transport", Morton sorting).
#pragma once

#include "fs_host.cuh"

namespace fs {

constexpr int kMortonMaxDim = 8;
// quantisation bits per axis of a d-dimensional Morton code
__host__ __device__ constexpr int morton_bits(int d) { return d <= 3 ? 21 : 63 / d; }

// Workspace offsets of the sort's buffers (box, keys, values, histograms).
struct MortonBufs {
    size_t box, keys0, keys1, vals0, vals1, hist;
};

void layout_morton(Layout& L, MortonBufs& M, int64_t n, int64_t m, int d);

// perm_x[i]: the caller's index of X's i-th point in Morton order (likewise
// perm_y for Y); 1 <= d <= kMortonMaxDim, device arrays, on c.stream.
fs_status morton_permutation(Call& c, const MortonBufs& M, const float* X, int64_t n,
                             const float* Y, int64_t m, int d, int* perm_x, int* perm_y);

}  // namespace fs

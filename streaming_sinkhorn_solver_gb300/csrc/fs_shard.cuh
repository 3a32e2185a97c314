// Row shards of a half-update.
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 1: the
// f-update of row i needs only x_i, a_i and the whole other side (Y, b, g),
// and symmetrically for the g-update, so a half-update partitions by rows of
// the updated side with no exchange inside it; G GPUs would each update their
// own rows and all-gather the potential before the next half.
//
// The updated side's rows are cut into `shards` contiguous ranges of whole
// units (the kernels' row blocks, so that every row keeps its position in its
// block and its arithmetic): shard s owns units [s U / G, (s + 1) U / G) of
// the U = ceil(rows / unit) units, clipped to the rows.  Shards are balanced
// to one unit and empty when G > U.
#pragma once

#include <stdint.h>

namespace fs {

inline void shard_range(int64_t rows, int64_t unit, int64_t shards, int64_t s, int64_t* r0,
                        int64_t* r1) {
    const int64_t units = (rows + unit - 1) / unit;
    const int64_t u0 = units * s / shards, u1 = units * (s + 1) / shards;
    *r0 = u0 * unit < rows ? u0 * unit : rows;
    *r1 = u1 * unit < rows ? u1 * unit : rows;
}

// Shard units of the two paths (rows per row block of their half-update).
int64_t shard_unit_fma(int32_t d);
int64_t shard_unit_tc();

}  // namespace fs

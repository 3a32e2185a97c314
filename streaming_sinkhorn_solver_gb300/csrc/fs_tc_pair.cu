// Fused half-update on CTA pairs: tcgen05.mma.cta_group::2 with M = 256
// (the pair's two 128-row tiles of Q) and N = 256 columns of K.
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 1
// (Proposition 1) and Method 2 (streaming kernels, row-stationary traversal,
// online max/sum-exp, fused write-back) -- the same computation as
// fs_tc_half.cu, mapped onto two SMs.
//
// Why pairs.  With one CTA, an M = N = 128 MMA step reads 4 KB of A and 4 KB
// of B from shared memory and the bulk copies write another 4 KB of B: about
// 192 B/clk at the f16 MMA rate, well above the ~128 B/clk an SM's shared
// memory delivers.  In a pair each SM keeps its own 128 Q rows and supplies
// half of each 256-row K tile, so an MMA step costs it 4 KB of A, 4 KB of B
// read and 4 KB of B written per 128 clocks (~96 B/clk), and its copy ring
// covers twice the latency for the same bytes.
//
// Roles (320 threads per CTA with online maxima, 576 with reference offsets;
// clusters of 2 along x):
//   warp 0     producer, both CTAs: own Q tile once, then per 256-column tile
//              the 1 KB bias slice and its own 128-row half of every K chunk,
//              the Q and K copies completing their bytes on the even CTA's
//              barriers (the even producer's expect_tx covers both halves);
//   warp 1     even CTA: issues the pair MMAs into TMEM buffer t mod 2 and
//              commits with multicast to both CTAs' barriers; odd CTA: only
//              allocates and frees the pair's TMEM with the even one;
//   warps 2-   epilogue groups, one thread per row, releasing TMEM buffers
//              to the even CTA's barrier (local and remote arrivals):
//              online mode: two groups, tile t going to group t mod 2, a
//              thread reading its 256 scores in two halves and folding them
//              into a running max and sum;
//              reference mode: kPairRefGroups groups spread over the two
//              TMEM buffers, each owning an equal share of a buffer's
//              columns: the group pre-loads its accumulators with
//              -M / kappa' (M = the row's previous LSE), then streams its
//              share in 32-column slices and only sums 2^{acc kappa' + bias}.
// Bias slices go through a ring of 8, so the producer never waits on them
// before issuing K chunks.
#include "fs_tc.cuh"

namespace fs {
namespace tc {

namespace {

constexpr int BNP = 256;                    // columns of a pair score tile
constexpr int kPairBufs = 2;                // TMEM buffers of BNP columns
constexpr int kPairTmemCols = kPairBufs * BNP;
constexpr int kPairBiasBytes = BNP * 4;
constexpr int kPairBiasSlots = 8;
constexpr int kPairMaxGroups = kPairRefGroups > kHalfGroups ? kPairRefGroups : kHalfGroups;

__host__ __device__ constexpr int pair_fixed_bytes(int nch, bool qres) {
    return 1024 + (qres ? nch * CHUNK_BYTES : 0) + kPairBiasSlots * kPairBiasBytes +
           BM * 8 * (kPairMaxGroups - 1) +
           8 * (2 * kMaxStages + 2 * kPairBufs + 2 * kPairBiasSlots + 2) + 16;
}

template <int GROUPS>
__device__ __forceinline__ void epi_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(GROUPS * kEpiWarps * 32) : "memory");
}

// One 32-column slice in reference mode: acc[] += 2^{v kappa' + bias}.
__device__ __forceinline__ void ref_slice(const float (&v)[32], const float4* __restrict__ sb,
                                          uint64_t ks2, uint64_t (&acc)[4]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 bb = sb[q];
        float x0, x1, x2, x3;
        upk(fma2(pk(v[4 * q], v[4 * q + 1]), ks2, pk(bb.x, bb.y)), x0, x1);
        upk(fma2(pk(v[4 * q + 2], v[4 * q + 3]), ks2, pk(bb.z, bb.w)), x2, x3);
        acc[(2 * q) & 3] = add2(acc[(2 * q) & 3], pk(ex2(x0), ex2(x1)));
        acc[(2 * q + 1) & 3] = add2(acc[(2 * q + 1) & 3], pk(ex2(x2), ex2(x3)));
    }
}

// one row's 128 scores: s = acc kappa' + bias, folded into (M, S)
__device__ __forceinline__ void fold128(float* v, const float4* sb, uint64_t ks2, float& M,
                                        float& S) {
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int q = 0; q < 32; ++q) {
        const float4 bb = sb[q];
        upk(fma2(pk(v[4 * q], v[4 * q + 1]), ks2, pk(bb.x, bb.y)), v[4 * q], v[4 * q + 1]);
        upk(fma2(pk(v[4 * q + 2], v[4 * q + 3]), ks2, pk(bb.z, bb.w)), v[4 * q + 2], v[4 * q + 3]);
        mx0 = max3(mx0, v[4 * q], v[4 * q + 1]);
        mx1 = max3(mx1, v[4 * q + 2], v[4 * q + 3]);
    }
    const float mx = fmaxf(mx0, mx1);
    if (mx > M) {
        S *= ex2(M - mx);
        M = mx;
    }
    if (M == -INFINITY) return;   // only padding columns so far: nothing to add
    const uint64_t nm = pk(-M, -M);
    uint64_t acc0 = pk(0.f, 0.f), acc1 = pk(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 32; ++q) {
        float x0, x1, x2, x3;
        upk(add2(pk(v[4 * q], v[4 * q + 1]), nm), x0, x1);
        upk(add2(pk(v[4 * q + 2], v[4 * q + 3]), nm), x2, x3);
        acc0 = add2(acc0, pk(ex2(x0), ex2(x1)));
        acc1 = add2(acc1, pk(ex2(x2), ex2(x3)));
    }
    float s0, s1, s2, s3;
    upk(acc0, s0, s1);
    upk(acc1, s2, s3);
    S += (s0 + s1) + (s2 + s3);
}

// Launch order.  The grid is one-dimensional, row_tiles * splits CTAs, and
// blocks start roughly in index order.  Consecutive pairs are taken in groups
// of raster_pairs row-tile pairs (the last group may be shorter); a group runs
// every column split of its pairs before the next group starts, so its Q tiles
// are reused from L2 by the later splits instead of being read again from
// DRAM once every row tile of a split has streamed past.
__device__ __forceinline__ void pair_tile(int splits, int raster_pairs, int64_t& rt, int& split) {
    // gridDim.x < 2^31 (checked at launch), so every quantity fits 32 bits
    const uint32_t pairs = gridDim.x / (2u * (uint32_t)splits);
    const uint32_t grp = raster_pairs > 0 ? min((uint32_t)raster_pairs, pairs) : pairs;
    const uint32_t L = blockIdx.x >> 1;
    const uint32_t g = L / (grp * (uint32_t)splits);
    const uint32_t base = g * grp;
    const uint32_t in_group = min(grp, pairs - base);
    const uint32_t w = L - g * grp * (uint32_t)splits;
    split = (int)(w / in_group);
    rt = 2 * (int64_t)(base + (w - (uint32_t)split * in_group)) + (blockIdx.x & 1);
}

}  // namespace

int pair_stages(int nch, bool qres) {
    const int stage = qres ? CHUNK_BYTES : 2 * CHUNK_BYTES;
    const int s = (kSmemLimit - pair_fixed_bytes(nch, qres)) / stage;
    return s < kMaxStages ? s : kMaxStages;
}

size_t pair_smem_bytes(int nch, bool qres, int stages) {
    const size_t stage = qres ? CHUNK_BYTES : 2 * CHUNK_BYTES;
    return (size_t)pair_fixed_bytes(nch, qres) + (size_t)stages * stage;
}

// a.col_tiles and a.tiles_per_split count 256-column tiles; a.K holds an even
// number of 128-row tiles; a.cbias has 256 entries per column tile.
template <bool QRES, bool REF>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(half_threads(REF), 1)
    k_half_pair(const __grid_constant__ TensorMap128 tmQ, const __grid_constant__ TensorMap128 tmK,
                TcHalfArgs a) {
    constexpr int GROUPS = REF ? kPairRefGroups : kHalfGroups;
    static_assert(!REF || GROUPS % kPairBufs == 0, "reference mode: equal groups per TMEM buffer");
    // reference mode: groups per TMEM buffer, columns of one group's share
    constexpr int SHARES = REF ? GROUPS / kPairBufs : 1;
    constexpr int SHARE_COLS = BNP / SHARES;
    static_assert(SHARE_COLS % 64 == 0, "a share is an even number of 32-column slices");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    int64_t rt;
    int split;
    pair_tile(a.splits, a.raster_pairs, rt, split);
    const int j0 = split * a.tiles_per_split;
    const int j1 = min(a.col_tiles, j0 + a.tiles_per_split);
    const int ntiles = j1 - j0;
    const int nch = a.nch;
    const int stages = a.stages;

    constexpr int STAGE_BYTES = QRES ? CHUNK_BYTES : 2 * CHUNK_BYTES;
    uint8_t* sQ = smem;
    uint8_t* sStage = smem + (QRES ? nch * CHUNK_BYTES : 0);
    uint8_t* sBias = sStage + stages * STAGE_BYTES;
    float2* sMerge = reinterpret_cast<float2*>(sBias + kPairBiasSlots * kPairBiasBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(sMerge + BM * (kPairMaxGroups - 1));
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;
    uint64_t* tempty = tfull + kPairBufs;
    uint64_t* bfull = tempty + kPairBufs;
    uint64_t* bempty = bfull + kPairBiasSlots;
    uint64_t* qfull = bempty + kPairBiasSlots;
    uint64_t* drain = qfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

    if (threadIdx.x == 0) {
        // the even CTA's full/qfull collect the bytes of both CTAs' copies (the
        // even producer's expect_tx covers both); its tempty also counts the
        // odd CTA's epilogue warps.  The odd CTA's full/qfull stay unused.
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        // a TMEM buffer is released by every epilogue warp that reads it, in
        // both CTAs: one group per CTA (online), SHARES (reference)
        constexpr int readers = SHARES * kEpiWarps;
        for (int b = 0; b < kPairBufs; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 2 * readers);
        }
        for (int b = 0; b < kPairBiasSlots; ++b) {
            mbar_init(&bfull[b], 1);
            mbar_init(&bempty[b], readers);
        }
        mbar_init(qfull, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    cluster_sync();   // every barrier of both CTAs exists before any remote arrival
    if (warp == 1) tmem_alloc_pair(tmem_slot, kPairTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer (both CTAs) ----------------
        if (lane == 0) {
            // both CTAs' copies complete their bytes on the even CTA's barriers
            const uint32_t qfull_lead = mapa_shared(smem_u32(qfull), 0);
            const uint32_t qrow0 = (uint32_t)(rt * nch) * BM;
            // L2 priorities with resident Q: the pairs running at once stream
            // the same K tiles, which are kept, while a Q tile is read once per
            // pair and goes first.  A streamed Q tile is re-read for every
            // column tile, so without resident Q neither operand is hinted.
            const uint64_t keep = l2_evict_last();
            if (QRES) {
                const uint64_t once = l2_evict_first();
                if (leader) mbar_arrive_expect_tx(qfull, (uint32_t)(2 * nch * CHUNK_BYTES));
                for (int c = 0; c < nch; ++c)
                    tma_chunk_pair_hint(sQ + c * CHUNK_BYTES, &tmQ, qrow0 + c * BM, qfull_lead, once);
            }
            int s = 0, issued = 0, bissued = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = 0; t < ntiles && ok; ++t) {
                const int b = t % kPairBiasSlots;
                if (!mbar_wait(&bempty[b], (uint32_t)((t / kPairBiasSlots) & 1) ^ 1u, a.err,
                               ERR_TIMEOUT_PRODUCER)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bfull[b], kPairBiasBytes);
                bulk_g2s(sBias + b * kPairBiasBytes, a.cbias + (int64_t)(j0 + t) * BNP,
                         kPairBiasBytes, &bfull[b]);
                ++bissued;
                const uint32_t krow0 = (uint32_t)((2 * (j0 + t) + (int)rank) * nch) * BM;
                for (int c = 0; c < nch; ++c) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, a.err, ERR_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = sStage + s * STAGE_BYTES;
                    const uint32_t full_lead = mapa_shared(smem_u32(&full[s]), 0);
                    if (leader) mbar_arrive_expect_tx(&full[s], 2 * STAGE_BYTES);
                    if (QRES) tma_chunk_pair_hint(st, &tmK, krow0 + c * BM, full_lead, keep);
                    else tma_chunk_pair(st, &tmK, krow0 + c * BM, full_lead);
                    if (!QRES) tma_chunk_pair(st + CHUNK_BYTES, &tmQ, qrow0 + c * BM, full_lead);
                    ++issued;
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let the copies already issued land before the pair can exit: the
                // even CTA's barriers count both CTAs' bytes, and the final cluster
                // barrier holds the odd CTA until the even one has drained them
                if (leader) {
                    int s2 = 0;
                    uint32_t ph2 = 0;
                    const int skip = issued > stages ? issued - stages : 0;
                    for (int i = 0; i < issued; ++i) {
                        if (i >= skip) mbar_wait_cluster(&full[s2], ph2, a.err, ERR_TIMEOUT_PRODUCER);
                        if (++s2 == stages) {
                            s2 = 0;
                            ph2 ^= 1u;
                        }
                    }
                    if (QRES) mbar_wait_cluster(qfull, 0, a.err, ERR_TIMEOUT_PRODUCER);
                }
                for (int i = bissued > kPairBiasSlots ? bissued - kPairBiasSlots : 0; i < bissued; ++i)
                    mbar_wait(&bfull[i % kPairBiasSlots], (uint32_t)((i / kPairBiasSlots) & 1), a.err,
                              ERR_TIMEOUT_PRODUCER);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (even CTA) ----------------
            constexpr uint32_t idesc = idesc_f16_f32(2 * BM, BNP);
            bool ok = true;
            if (QRES) ok = mbar_wait_cluster(qfull, 0, a.err, ERR_TIMEOUT_MMA);
            tc_fence_after();
            int s = 0;
            uint32_t ph = 0;
            // online: use u of a buffer waits for the release of use u - 1 (the
            // first passes at once); reference: the epilogue releases every
            // buffer once before its first use, after pre-loading it
            for (int t = 0; t < ntiles && ok; ++t) {
                const int b = t & 1;
                if (!mbar_wait_cluster(&tempty[b], (uint32_t)((t >> 1) & 1) ^ (REF ? 0u : 1u), a.err,
                                       ERR_TIMEOUT_MMA)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(b * BNP);
                for (int c = 0; c < nch; ++c) {
                    if (!mbar_wait_cluster(&full[s], ph, a.err, ERR_TIMEOUT_MMA)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* st = sStage + s * STAGE_BYTES;
                    const uint32_t aaddr = smem_u32(QRES ? sQ + c * CHUNK_BYTES : st + CHUNK_BYTES);
                    const uint32_t baddr = smem_u32(st);
                    // the start-address field counts 16-byte units: a 32-byte step is + 2
                    const uint64_t ad0 = sdesc_sw128(aaddr), bd0 = sdesc_sw128(baddr);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16_pair(d_tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc, REF || (c | kk) != 0);
                    mma_commit_pair(&empty[s], 3);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair(&tfull[b], 3);
            }
            mma_commit_pair(drain, 3);
            mbar_wait(drain, 0, a.err, ERR_TIMEOUT_MMA);
        }
    } else {
        // ---------------- epilogue groups: one thread per row ----------------
        const int grp = (warp - 2) / kEpiWarps;
        const int quarter = warp & 3;
        const int rloc = quarter * 32 + lane;
        const int64_t row = rt * BM + rloc;
        const float ks = *a.kscale;
        const uint64_t ks2 = pk(ks, ks);
        const uint32_t lofs = (uint32_t)(quarter * 32) << 16;
        float M = -INFINITY, S = 0.f;
        if constexpr (REF) {
            // group g: TMEM buffer g / SHARES (tiles t = that mod 2), column
            // share g % SHARES
            constexpr int SLICES = SHARE_COLS / 32;
            const int b = grp / SHARES, h = grp % SHARES;
            const int64_t rr = row < a.nr ? row : a.nr - 1;
            M = a.rlogw2[rr] - a.rbias[rr];
            const float fill = __fdividef(-M, ks);   // the offset only has to be M up to rounding
            const uint32_t buf = tmem + (uint32_t)(b * BNP + h * SHARE_COLS) + lofs;
            const uint32_t tempty_lead = mapa_shared(smem_u32(&tempty[b]), 0);
#pragma unroll
            for (int q = 0; q < 4 * SLICES; ++q) tmem_fill8(buf + q * 8, fill);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(tempty_lead);
            uint64_t acc[4] = {pk(0.f, 0.f), pk(0.f, 0.f), pk(0.f, 0.f), pk(0.f, 0.f)};
            for (int t = b; t < ntiles; t += kPairBufs) {
                if (!mbar_wait_cluster(&tfull[b], (uint32_t)((t >> 1) & 1), a.err, ERR_TIMEOUT_EPILOGUE))
                    break;
                tc_fence_after();
                const int bs = t % kPairBiasSlots;
                if (!mbar_wait(&bfull[bs], (uint32_t)((t / kPairBiasSlots) & 1), a.err,
                               ERR_TIMEOUT_EPILOGUE))
                    break;
                const float4* sb = reinterpret_cast<const float4*>(sBias + bs * kPairBiasBytes) +
                                   h * (SHARE_COLS / 4);
                // slice q + 1 loads while slice q is summed; va holds the even
                // slices, vb the odd ones.  The loop stays rolled: unrolled,
                // the bias loads of later slices move up and spill registers.
                float va[32], vb[32];
                tmem_ld32(buf, va);
                tmem_wait_ld();
                tmem_reg_fence(va);
#pragma unroll 1
                for (int q = 0; q < SLICES; q += 2) {
                    tmem_ld32(buf + (q + 1) * 32, vb);
                    ref_slice(va, sb + q * 8, ks2, acc);
                    tmem_wait_ld();
                    tmem_reg_fence(vb);
                    if (q + 2 < SLICES) {
                        tmem_ld32(buf + (q + 2) * 32, va);
                        ref_slice(vb, sb + (q + 1) * 8, ks2, acc);
                        tmem_wait_ld();
                        tmem_reg_fence(va);
                    }
                }
                // the share is in registers: pre-load it again, hand it back
#pragma unroll
                for (int q = 0; q < 4 * SLICES; ++q) tmem_fill8(buf + q * 8, fill);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(tempty_lead);
                ref_slice(vb, sb + (SLICES - 1) * 8, ks2, acc);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bempty[bs]);
            }
            float s0, s1, s2, s3, s4, s5, s6, s7;
            upk(acc[0], s0, s1);
            upk(acc[1], s2, s3);
            upk(acc[2], s4, s5);
            upk(acc[3], s6, s7);
            S = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
        } else {
            for (int t = grp; t < ntiles; t += GROUPS) {
                const int b = t & 1;
                const uint32_t ph = (uint32_t)((t >> 1) & 1);
                if (!mbar_wait_cluster(&tfull[b], ph, a.err, ERR_TIMEOUT_EPILOGUE)) break;
                tc_fence_after();
                const int bs = t % kPairBiasSlots;
                if (!mbar_wait(&bfull[bs], (uint32_t)((t / kPairBiasSlots) & 1), a.err,
                               ERR_TIMEOUT_EPILOGUE))
                    break;
                const float4* sb = reinterpret_cast<const float4*>(sBias + bs * kPairBiasBytes);
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    float v[128];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld32(tmem + (uint32_t)(b * BNP + h * 128) + lofs + q * 32, v + q * 32);
                    tmem_wait_ld();
                    tmem_reg_fence(v);
                    if (h == 1) {
                        // both halves are in registers: hand the buffer back to the MMA
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&tempty[b]), 0));
                    }
                    fold128(v, sb + h * 32, ks2, M, S);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bempty[bs]);
            }
        }

        // merge the groups in a fixed order: group 0 absorbs groups 1, 2, ...
        if (grp > 0) sMerge[(grp - 1) * BM + rloc] = make_float2(M, S);
        epi_bar_sync<GROUPS>();
        if (grp == 0) {
            float Mt = M, St = S;
#pragma unroll
            for (int g = 1; g < GROUPS; ++g) {
                const float2 o = sMerge[(g - 1) * BM + rloc];
                const float Mn = fmaxf(Mt, o.x);
                // a group that saw only padding has (M, S) = (-inf, 0) and adds nothing
                St = (Mt == -INFINITY ? 0.f : St * ex2(Mt - Mn)) +
                     (o.x == -INFINITY ? 0.f : o.y * ex2(o.x - Mn));
                Mt = Mn;
            }
            if (row < a.nr) {
                if (a.splits > 1) {
                    a.partial[(int64_t)split * a.nr + row] = make_float2(Mt, St);
                } else {
                    if (REF && !(St >= kTcMinRefSum && St <= kTcMaxRefSum)) {
                        const unsigned int slot = atomicAdd(&a.fix_count[0], 1u);
                        if (slot < (unsigned int)a.nr) a.fix_list[slot] = (int)row;
                    }
                    const float lse2 = Mt + log2f(St);
                    if (a.rnorm != nullptr) {
                        a.pot[row] = a.rnorm[row] - a.eps_ln2 * lse2;
                        a.rbias[row] = a.rlogw2[row] - lse2;
                    } else {
                        a.pot[row] = lse2;
                    }
                }
            }
        }
    }

    // no MMA of the pair is in flight past this point (the even CTA drained
    // them); neither CTA frees TMEM or leaves while the other may still use it
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kPairTmemCols);
    }
}

template <bool QRES, bool REF>
cudaError_t launch_half_pair_t(const TcHalfArgs& a, const TensorMap128& tmQ, const TensorMap128& tmK,
                               int row_tiles, size_t smem, cudaStream_t s) {
    const cudaError_t e = cudaFuncSetAttribute(
        k_half_pair<QRES, REF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((int64_t)row_tiles * a.splits));
    k_half_pair<QRES, REF><<<grid, half_threads(REF), smem,
                             s>>>(tmQ, tmK, a);
    return cudaGetLastError();
}

cudaError_t launch_half_pair(const TcHalfArgs& a, const TensorMap128& tmQ,
                             const TensorMap128& tmK, int row_tiles, bool qres, cudaStream_t s) {
    if (row_tiles % 2 != 0 || a.splits < 1 || (int64_t)row_tiles * a.splits > 0x7fffffff)
        return cudaErrorInvalidValue;
    const size_t smem = pair_smem_bytes(a.nch, qres, a.stages);
    cudaError_t e;
    if (a.use_ref)
        e = qres ? launch_half_pair_t<true, true>(a, tmQ, tmK, row_tiles, smem, s)
                 : launch_half_pair_t<false, true>(a, tmQ, tmK, row_tiles, smem, s);
    else
        e = qres ? launch_half_pair_t<true, false>(a, tmQ, tmK, row_tiles, smem, s)
                 : launch_half_pair_t<false, false>(a, tmQ, tmK, row_tiles, smem, s);
    count_launch();
    return e;
}

}  // namespace tc
}  // namespace fs

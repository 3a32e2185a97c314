// Reference-offset half-update on the tcgen05 tensor cores (one CTA per
// 128-row tile, d <= 128).
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 1
// (Proposition 1: the f-update is a row LSE of the biased dot-product score
// matrix (Q K^T + bias)/eps) and Method 2 (streaming kernels and tiling: a Q
// row block stays on chip while every K block streams past; score, bias,
// exponent, sum and potential write-back fused in one pass).
//
// Once the potentials have settled, a row's previous LSE is a fixed exponent
// offset M for the whole pass: no running max.  The offset enters the
// accumulator through the tensor core: one more K = 16 step per tile
// multiplies an offset column block of the resident Q tile, whose first two
// columns hold the fp16 split (hi, lo) of -M / (ks 2^p) for each row, by a
// constant column block whose first two columns hold 2^p, so the
// accumulator is Q K^T - M / ks and every score costs one multiply-add, one
// exp2 and one add (packed two by two).  The offset actually applied is
// M' = -(hi + lo) 2^p ks, which the write-back uses; 2^p puts the CTA's
// largest |M| / ks near 2^14, inside fp16.  The row's sum is range-checked at
// the end; a row outside the range goes to the fixup list.
//
// One CTA owns a 128-row tile of Q (resident in shared memory) and a range
// of 128-column tiles of K; tile t lives in TMEM buffer t mod 4.
//   warp 0     producer: Q once; per tile its 512-byte bias slice (a ring of
//              16) and its K tile into K slot t mod 4, all with cp.async.bulk;
//   warp 1     one thread issues the tile's tcgen05.mma (M = 128, N = 128,
//              K = 16 steps) and one commit;
//   warps 2-17 four epilogue groups of four warps, group g owning buffer g
//              and the tiles t = g (mod 4).
// The epilogue reads the scores in the 16x256b shape, in which a thread holds
// two columns of every eight for two rows of a 16-lane block, so that over its
// warp's 32 lanes it covers 4 rows x 32 columns of a tile (rather than 1 row
// x 128 columns).  Every bias value it loads from shared memory then serves
// four rows: per-thread broadcast loads of a per-column bias would otherwise
// cost as much shared-memory bandwidth (128 bytes per clock and SM) as the
// exponentials cost MUFU time.  The four threads sharing a row add their
// sums once, at the end.
// The K slots are tied to the TMEM buffers so that the MMA thread, whose
// serial work per tile bounds the kernel once the epilogue is cheap, waits on
// a single barrier per tile: tempty[b] completes when the group has released
// buffer b (four arrivals), the producer has armed it (one arrival with the
// K tile's byte count) and the K tile has landed.  The producer re-uses slot
// b once the MMAs of the tile before have completed (tfull[b]), so the MMA
// thread commits once per tile.  Its descriptors are formed before the loop;
// a K step is a 32-byte advance of both start addresses.
#include "fs_tc.cuh"

namespace fs {
namespace tc {

namespace {

constexpr int kRefThreads = 32 * (2 + kRefGroups * kEpiWarps);
constexpr int kRefBiasSlots = 16;
constexpr int kBiasBytes = BN * 4;
static_assert(kRefGroups == kTmemBufs, "one epilogue group per TMEM buffer");

__host__ __device__ constexpr int ref_smem_bytes(int nch) {
    return 1024 /* alignment slack */ + (1 + kTmemBufs) * nch * CHUNK_BYTES +
           2 * CHUNK_BYTES /* offset column blocks */ + kRefBiasSlots * kBiasBytes +
           BM * 4 * (kRefGroups - 1) /* group merge */ +
           8 * (1 + 2 * kTmemBufs + 2 * kRefBiasSlots + 2) + 16;
}

// fp16 split of the scaled row offset: hi + lo = -M / (ks 2^p) to about 22
// bits (clamped inside the fp16 range: a row clamped here leaves the guarded
// range and is recomputed by the fixup)
__device__ __forceinline__ void offset_split(float M, float inv_scale, __half& hi, __half& lo) {
    const float t = fminf(fmaxf(-M * inv_scale, -60000.f), 60000.f);
    hi = __float2half_rn(t);
    lo = __float2half_rn(t - __half2float(hi));
}

// the offset the accumulator received: -(hi + lo) 2^p ks
__device__ __forceinline__ float offset_applied(__half hi, __half lo, float scale) {
    return -(__half2float(hi) + __half2float(lo)) * scale;
}

// One 16-lane x 32-column slice (tmem_ld16x32 layout): for each repetition
// i, the column pair's bias bp[i] serves both rows; lo/hi accumulate the rows
// t/4 and t/4 + 8 of the block: acc += 2^{v kappa' + bias} (v already holds
// the row's -M' / kappa').
__device__ __forceinline__ void ref_slice(const float (&v)[16], const uint64_t (&bp)[4],
                                          uint64_t ks2, uint64_t& lo, uint64_t& hi) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float x0, x1, x2, x3;
        upk(fma2(pk(v[4 * i], v[4 * i + 1]), ks2, bp[i]), x0, x1);
        upk(fma2(pk(v[4 * i + 2], v[4 * i + 3]), ks2, bp[i]), x2, x3);
        lo = add2(lo, pk(ex2(x0), ex2(x1)));
        hi = add2(hi, pk(ex2(x2), ex2(x3)));
    }
}

template <int NCH>
__global__ void __launch_bounds__(kRefThreads, 1) k_half_ref(TcHalfArgs a) {
    constexpr int TILE_BYTES = NCH * CHUNK_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rt = blockIdx.x;
    const int j0 = blockIdx.y * a.tiles_per_split;
    const int ntiles = min(a.col_tiles, j0 + a.tiles_per_split) - j0;

    uint8_t* sQ = smem;
    uint8_t* sK = smem + TILE_BYTES;                       // slot b at sK + b * TILE_BYTES
    uint8_t* sQx = sK + kTmemBufs * TILE_BYTES;            // offset column block of Q
    uint8_t* sKx = sQx + CHUNK_BYTES;                      // constant column block of K
    uint8_t* sBias = sKx + CHUNK_BYTES;
    float* sMerge = reinterpret_cast<float*>(sBias + kRefBiasSlots * kBiasBytes);
    uint64_t* qfull = reinterpret_cast<uint64_t*>(sMerge + BM * (kRefGroups - 1));
    uint64_t* tfull = qfull + 1;                 // MMAs of the buffer's tile complete
    uint64_t* tempty = tfull + kTmemBufs;        // buffer released and its K tile landed
    uint64_t* bfull = tempty + kTmemBufs;
    uint64_t* bempty = bfull + kRefBiasSlots;
    uint64_t* drain = bempty + kRefBiasSlots;
    uint64_t* xfull = drain + 1;                 // offset column blocks written
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xfull + 1);
    uint32_t* sMmax = tmem_slot + 1;             // largest |M| of the tile's rows (float bits)

    if (threadIdx.x == 0) {
        mbar_init(qfull, 1);
        for (int b = 0; b < kTmemBufs; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps + 1);
        }
        for (int s = 0; s < kRefBiasSlots; ++s) {
            mbar_init(&bfull[s], 1);
            mbar_init(&bempty[s], kEpiWarps);
        }
        mbar_init(drain, 1);
        mbar_init(xfull, kRefGroups * kEpiWarps);
        *sMmax = 0u;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            mbar_arrive_expect_tx(qfull, (uint32_t)TILE_BYTES);
            const char* Qg = reinterpret_cast<const char*>(a.Q) + rt * (int64_t)TILE_BYTES;
#pragma unroll
            for (int c = 0; c < NCH; ++c)
                bulk_g2s(sQ + c * CHUNK_BYTES, Qg + c * CHUNK_BYTES, CHUNK_BYTES, qfull);
            const char* Kg = reinterpret_cast<const char*>(a.K) + (int64_t)j0 * TILE_BYTES;
            int kiss = 0, biss = 0;
            bool ok = true;
            for (int t = 0; t < ntiles; ++t) {
                const int bs = t % kRefBiasSlots;
                ok = mbar_wait(&bempty[bs], (uint32_t)((t / kRefBiasSlots) & 1) ^ 1u, a.err,
                               ERR_TIMEOUT_PRODUCER);
                if (!ok) break;
                mbar_arrive_expect_tx(&bfull[bs], kBiasBytes);
                bulk_g2s(sBias + bs * kBiasBytes, a.cbias + (int64_t)(j0 + t) * BN, kBiasBytes,
                         &bfull[bs]);
                biss = t + 1;
                const int b = t & (kTmemBufs - 1);
                const int u = t >> 2;
                // slot b is free once the MMAs of tile t - 4 have completed
                if (u > 0) {
                    ok = mbar_wait(&tfull[b], (uint32_t)((u - 1) & 1), a.err, ERR_TIMEOUT_PRODUCER);
                    if (!ok) break;
                }
                uint8_t* slot = sK + b * TILE_BYTES;
                mbar_arrive_expect_tx(&tempty[b], (uint32_t)TILE_BYTES);
#pragma unroll
                for (int c = 0; c < NCH; ++c)
                    bulk_g2s(slot + c * CHUNK_BYTES, Kg + (int64_t)t * TILE_BYTES + c * CHUNK_BYTES,
                             CHUNK_BYTES, &tempty[b]);
                kiss = t + 1;
            }
            if (!ok) {
                // let every copy already issued land before the CTA can exit
                for (int t = kiss > kTmemBufs ? kiss - kTmemBufs : 0; t < kiss; ++t)
                    mbar_wait(&tempty[t & (kTmemBufs - 1)], (uint32_t)((t >> 2) & 1), a.err,
                              ERR_TIMEOUT_PRODUCER);
                for (int t = biss > kRefBiasSlots ? biss - kRefBiasSlots : 0; t < biss; ++t)
                    mbar_wait(&bfull[t % kRefBiasSlots], (uint32_t)((t / kRefBiasSlots) & 1),
                              a.err, ERR_TIMEOUT_PRODUCER);
            }
            mbar_wait(qfull, 0, a.err, ERR_TIMEOUT_PRODUCER);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            uint64_t qd[NCH];
#pragma unroll
            for (int c = 0; c < NCH; ++c) qd[c] = sdesc_sw128(smem_u32(sQ + c * CHUNK_BYTES));
            const uint64_t kd0 = sdesc_sw128(smem_u32(sK));
            const uint64_t qxd = sdesc_sw128(smem_u32(sQx));
            const uint64_t kxd = sdesc_sw128(smem_u32(sKx));
            bool ok = mbar_wait(qfull, 0, a.err, ERR_TIMEOUT_MMA) &&
                      mbar_wait(xfull, 0, a.err, ERR_TIMEOUT_MMA);
            for (int t = 0; t < ntiles && ok; ++t) {
                const int b = t & (kTmemBufs - 1);
                if (!mbar_wait(&tempty[b], (uint32_t)((t >> 2) & 1), a.err, ERR_TIMEOUT_MMA)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(b * BN);
                const uint64_t kd = kd0 + (uint64_t)((b * TILE_BYTES) >> 4);
#pragma unroll
                for (int c = 0; c < NCH; ++c)
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16(d_tmem, qd[c] + (uint64_t)(2 * kk),
                                kd + (uint64_t)((c * CHUNK_BYTES) >> 4) + (uint64_t)(2 * kk), idesc,
                                (c | kk) != 0);
                mma_f16(d_tmem, qxd, kxd, idesc, 1);      // + (-M / ks) for every row
                mma_commit(&tfull[b]);
            }
            // every MMA issued has completed once `drain` fires
            mma_commit(drain);
            mbar_wait(drain, 0, a.err, ERR_TIMEOUT_MMA);
        }
    } else {
        // ---------------- epilogue groups ----------------
        const int grp = (warp - 2) / kEpiWarps;
        const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
        const float ks = *a.kscale;
        const uint64_t ks2 = pk(ks, ks);
        // The offset column blocks.  The tile's largest |M| (the warps of
        // group 0 cover its 128 rows) sets 2^p; then the 16 warps write the
        // 2 x 128 rows x 8 16-byte units of the two blocks.
        const int ew = warp - 2;                    // epilogue warp 0..15
        if (grp == 0) {
            float mabs = 0.f;
            const int64_t rk = min(rt * BM + quarter * 32 + lane, a.nr - 1);
            mabs = fabsf(a.rlogw2[rk] - a.rbias[rk]);
            if (!(mabs <= 3.0e38f)) mabs = 3.0e38f;   // NaN and inf: the largest finite
            const unsigned int mb = __reduce_max_sync(0xffffffffu, __float_as_uint(mabs));
            if (lane == 0) atomicMax(sMmax, mb);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kRefGroups * kEpiWarps * 32) : "memory");
        float scale, inv_scale;
        __half two_p;
        {
            const float q = __uint_as_float(*sMmax) / ks;
            int p = 0;
            if (q > 0.f && q <= 3.0e38f) p = min(max(ilogbf(q) - 13, -14), 15);
            two_p = __float2half_rn(ldexpf(1.f, p));
            scale = ldexpf(ks, p);
            inv_scale = 1.f / scale;
        }
        for (int idx = ew * 32 + lane; idx < 2 * BM * 8; idx += kRefGroups * kEpiWarps * 32) {
            const int blk = idx >> 10, r = (idx >> 3) & (BM - 1), u = idx & 7;
            __align__(16) __half h[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) h[q] = __float2half_rn(0.f);
            if (u == 0) {
                if (blk == 0) {
                    const int64_t rr = min(rt * BM + r, a.nr - 1);
                    offset_split(a.rlogw2[rr] - a.rbias[rr], inv_scale, h[0], h[1]);
                } else {
                    h[0] = two_p;
                    h[1] = two_p;
                }
            }
            *reinterpret_cast<uint4*>((blk ? sKx : sQx) + swz_offset(r, u * 8)) =
                *reinterpret_cast<const uint4*>(h);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(xfull);
        const uint32_t buf = tmem + (uint32_t)(grp * BN) + ((uint32_t)(quarter * 32) << 16);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[grp]);

        // rows of this thread: 32*quarter + lane/4 + 8k (k = 0..3; acc[k]),
        // columns 8i + 2(lane%4) + {0, 1} of every 32-column quarter
        const int cpair = 2 * (lane & 3);
        uint64_t acc[4] = {pk(0.f, 0.f), pk(0.f, 0.f), pk(0.f, 0.f), pk(0.f, 0.f)};
        for (int t = grp; t < ntiles; t += kRefGroups) {
            if (!mbar_wait(&tfull[grp], (uint32_t)((t >> 2) & 1), a.err, ERR_TIMEOUT_EPILOGUE))
                break;
            tc_fence_after();
            const int bs = t % kRefBiasSlots;
            if (!mbar_wait(&bfull[bs], (uint32_t)((t / kRefBiasSlots) & 1), a.err,
                           ERR_TIMEOUT_EPILOGUE))
                break;
            const uint64_t* sb =
                reinterpret_cast<const uint64_t*>(sBias + bs * kBiasBytes + cpair * 4);
            // slices s = 2 cq + h: column quarter cq, lane half h; the next
            // slice's load is in flight while one is summed, and the next
            // quarter's bias pairs while its second slice is
            float va[16], vb[16];
            uint64_t bp[4], bn[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) bp[i] = sb[(8 * i) / 2];
            tmem_ld16x32(buf, va);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int cq = s >> 1, h = s & 1;
                float(&cur)[16] = (s & 1) ? vb : va;
                float(&nxt)[16] = (s & 1) ? va : vb;
                tmem_wait_ld();
                tmem_reg_fence(cur);
                if (s < 7) {
                    const int s1 = s + 1;
                    tmem_ld16x32(buf + ((uint32_t)(16 * (s1 & 1)) << 16) + (uint32_t)(32 * (s1 >> 1)),
                                 nxt);
                } else {
                    // every score of the tile is in registers: release the buffer
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[grp]);
                }
                if (h == 1 && cq < 3) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) bn[i] = sb[(32 * (cq + 1) + 8 * i) / 2];
                }
                ref_slice(cur, bp, ks2, acc[2 * h], acc[2 * h + 1]);
                if (h == 1 && cq < 3) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) bp[i] = bn[i];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bempty[bs]);
        }
        // row sums: the pair halves, then the four threads sharing the rows
        float S4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float x, y;
            upk(acc[k], x, y);
            S4[k] = x + y;
            S4[k] += __shfl_xor_sync(0xffffffffu, S4[k], 1);
            S4[k] += __shfl_xor_sync(0xffffffffu, S4[k], 2);
        }
        // from here on a thread owns the row 32*quarter + lane/4 + 8(lane%4)
        const int kown = lane & 3;
        const float S = kown == 0 ? S4[0] : kown == 1 ? S4[1] : kown == 2 ? S4[2] : S4[3];
        const int rloc = quarter * 32 + (lane >> 2) + 8 * kown;
        const int64_t row = rt * BM + rloc;
        const int64_t rr = row < a.nr ? row : a.nr - 1;
        __half mhi, mlo;
        offset_split(a.rlogw2[rr] - a.rbias[rr], inv_scale, mhi, mlo);
        const float M = offset_applied(mhi, mlo, scale);
        // every group used the same offset M: the row sum is the groups'
        // sums, added in a fixed order
        if (grp > 0) sMerge[(grp - 1) * BM + rloc] = S;
        asm volatile("bar.sync 1, %0;" ::"n"(kRefGroups * kEpiWarps * 32) : "memory");
        if (grp == 0 && row < a.nr) {
            float St = S;
#pragma unroll
            for (int g = 1; g < kRefGroups; ++g) St += sMerge[(g - 1) * BM + rloc];
            if (a.splits > 1) {
                a.partial[(int64_t)blockIdx.y * a.nr + row] = make_float2(M, St);
            } else {
                if (!(St >= kTcMinRefSum && St <= kTcMaxRefSum)) {
                    const unsigned int slot = atomicAdd(&a.fix_count[0], 1u);
                    if (slot < (unsigned int)a.nr) a.fix_list[slot] = (int)row;
                }
                const float lse2 = M + log2f(St);
                a.pot[row] = a.rnorm[row] - a.eps_ln2 * lse2;
                a.rbias[row] = a.rlogw2[row] - lse2;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int NCH>
cudaError_t launch_ref_t(const TcHalfArgs& a, int row_tiles, cudaStream_t s) {
    constexpr int smem = ref_smem_bytes(NCH);
    static_assert(smem <= kSmemLimit, "reference kernel does not fit in shared memory");
    const cudaError_t e =
        cudaFuncSetAttribute(k_half_ref<NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k_half_ref<NCH><<<dim3((unsigned)row_tiles, (unsigned)a.splits), kRefThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_half_ref(const TcHalfArgs& a, int row_tiles, cudaStream_t s) {
    cudaError_t e;
    if (a.nch == 1)
        e = launch_ref_t<1>(a, row_tiles, s);
    else if (a.nch == 2)
        e = launch_ref_t<2>(a, row_tiles, s);
    else
        return cudaErrorInvalidValue;
    count_launch();
    return e;
}

}  // namespace tc
}  // namespace fs

// Fused half-update on the tcgen05 tensor cores (d > 16), online-max form.
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 1
// (Proposition 1: the f-update is a row LSE of the biased dot-product score
// matrix (Q K^T + bias)/eps) and Method 2 (streaming kernels and tiling: the
// n x m matrix never reaches HBM; a Q row block stays on chip while every K
// block streams past; running row max and sum-exp on chip; score, bias, LSE
// and potential write-back fused in one pass).
//
// One CTA owns a 128-row tile of Q and a range of 128-column tiles of K.
//   warp 0     producer: Q once (resident in shared memory up to d = 512,
//              otherwise streamed beside K), then for every column tile its
//              512-byte bias slice (a ring of 16) and its K chunks (128 x 64
//              fp16, 16 KB, pre-swizzled in HBM) into a ring sized to the free
//              space, all with cp.async.bulk;
//   warp 1     one thread issues tcgen05.mma (M = 128, N = 128, K = 16 steps)
//              into TMEM buffer t mod 4;
//   warps 2-9  two epilogue groups of four warps, tile t going to group
//              t mod 2; a thread owns one row, reads its 128 scores, forms
//              s = acc kappa' + bias (packed f32x2 FMA) and folds them into the
//              row's running max M and sum S of 2^{s-M}.
// At the end the groups' (M, S) are merged in a fixed order and the row
// potential and next bias are written (or (M, S) partials per split).  This
// kernel serves the first iterations and the log2-sum-exp pre-pass of the
// plan operators; settled iterations with d <= 128 use the reference-offset
// kernel (k_half_ref), which needs no running max.
#include "fs_tc.cuh"

namespace fs {
namespace tc {

namespace {

constexpr int kBiasBytes = BN * 4;
// Bias slices in flight: deeper than the K ring (in tiles), so the producer's
// wait for a free bias slot never holds back the next K chunks.
constexpr int kBiasSlots = 16;

__host__ __device__ constexpr int half_fixed_bytes(int nch, bool qres) {
    return 1024 /* alignment slack */ + (qres ? nch * CHUNK_BYTES : 0) + kBiasSlots * kBiasBytes +
           BM * 8 * (kHalfGroups - 1) /* group merge */ +
           8 * (2 * kMaxStages + 2 * kTmemBufs + 2 * kBiasSlots + 2) + 16;
}

template <int GROUPS>
__device__ __forceinline__ void epi_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(GROUPS * kEpiWarps * 32) : "memory");
}

}  // namespace

int half_stages(int nch, bool qres) {
    const int stage = qres ? CHUNK_BYTES : 2 * CHUNK_BYTES;
    const int s = (kSmemLimit - half_fixed_bytes(nch, qres)) / stage;
    return s < kMaxStages ? s : kMaxStages;
}

size_t half_smem_bytes(int nch, bool qres, int stages) {
    const size_t stage = qres ? CHUNK_BYTES : 2 * CHUNK_BYTES;
    return (size_t)half_fixed_bytes(nch, qres) + (size_t)stages * stage;
}

template <bool QRES>
__global__ void __launch_bounds__(kHalfThreads, 1) k_half_tc(TcHalfArgs a) {
    constexpr int GROUPS = kHalfGroups;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rt = blockIdx.x;
    const int j0 = blockIdx.y * a.tiles_per_split;
    const int j1 = min(a.col_tiles, j0 + a.tiles_per_split);
    const int ntiles = j1 - j0;
    const int nch = a.nch;
    const int stages = a.stages;

    constexpr int STAGE_BYTES = QRES ? CHUNK_BYTES : 2 * CHUNK_BYTES;
    uint8_t* sQ = smem;
    uint8_t* sStage = smem + (QRES ? nch * CHUNK_BYTES : 0);
    uint8_t* sBias = sStage + stages * STAGE_BYTES;
    float2* sMerge = reinterpret_cast<float2*>(sBias + kBiasSlots * kBiasBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(sMerge + BM * (kHalfGroups - 1));
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;
    uint64_t* tempty = tfull + kTmemBufs;
    uint64_t* bfull = tempty + kTmemBufs;
    uint64_t* bempty = bfull + kBiasSlots;
    uint64_t* qfull = bempty + kBiasSlots;
    uint64_t* drain = qfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < kTmemBufs; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
        }
        for (int b = 0; b < kBiasSlots; ++b) {
            mbar_init(&bfull[b], 1);
            mbar_init(&bempty[b], kEpiWarps);
        }
        mbar_init(qfull, 1);
        mbar_init(drain, 1);
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
            const char* Qg = reinterpret_cast<const char*>(a.Q) + rt * nch * (int64_t)CHUNK_BYTES;
            if (QRES) {
                mbar_arrive_expect_tx(qfull, (uint32_t)(nch * CHUNK_BYTES));
                for (int c = 0; c < nch; ++c)
                    bulk_g2s(sQ + c * CHUNK_BYTES, Qg + c * (int64_t)CHUNK_BYTES, CHUNK_BYTES, qfull);
            }
            int s = 0, issued = 0, bissued = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = 0; t < ntiles && ok; ++t) {
                const int b = t % kBiasSlots;
                if (!mbar_wait(&bempty[b], (uint32_t)((t / kBiasSlots) & 1) ^ 1u, a.err,
                               ERR_TIMEOUT_PRODUCER)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bfull[b], kBiasBytes);
                bulk_g2s(sBias + b * kBiasBytes, a.cbias + (int64_t)(j0 + t) * BN, kBiasBytes, &bfull[b]);
                ++bissued;
                const char* Kg =
                    reinterpret_cast<const char*>(a.K) + (int64_t)(j0 + t) * nch * CHUNK_BYTES;
                for (int c = 0; c < nch; ++c) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, a.err, ERR_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = sStage + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                    bulk_g2s(st, Kg + c * (int64_t)CHUNK_BYTES, CHUNK_BYTES, &full[s]);
                    if (!QRES)
                        bulk_g2s(st + CHUNK_BYTES, Qg + c * (int64_t)CHUNK_BYTES, CHUNK_BYTES,
                                 &full[s]);
                    ++issued;
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA can exit
                int s2 = 0;
                uint32_t ph2 = 0;
                const int skip = issued > stages ? issued - stages : 0;
                for (int i = 0; i < issued; ++i) {
                    if (i >= skip) mbar_wait(&full[s2], ph2, a.err, ERR_TIMEOUT_PRODUCER);
                    if (++s2 == stages) {
                        s2 = 0;
                        ph2 ^= 1u;
                    }
                }
                for (int i = bissued > kBiasSlots ? bissued - kBiasSlots : 0; i < bissued; ++i)
                    mbar_wait(&bfull[i % kBiasSlots], (uint32_t)((i / kBiasSlots) & 1), a.err,
                              ERR_TIMEOUT_PRODUCER);
                if (QRES) mbar_wait(qfull, 0, a.err, ERR_TIMEOUT_PRODUCER);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // Buffer use u waits for the epilogue's release of use u - 1 (the
        // first use passes at once).
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            bool ok = true;
            if (QRES) ok = mbar_wait(qfull, 0, a.err, ERR_TIMEOUT_MMA);
            tc_fence_after();
            int s = 0;
            uint32_t ph = 0;
            for (int t = 0; t < ntiles && ok; ++t) {
                const int b = t & (kTmemBufs - 1);
                const uint32_t use_ph = (uint32_t)((t >> 2) & 1) ^ 1u;
                if (!mbar_wait(&tempty[b], use_ph, a.err, ERR_TIMEOUT_MMA)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(b * BN);
                for (int c = 0; c < nch; ++c) {
                    if (!mbar_wait(&full[s], ph, a.err, ERR_TIMEOUT_MMA)) {
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
                        mma_f16(d_tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc, (c | kk) != 0);
                    mma_commit(&empty[s]);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[b]);
            }
            // every MMA issued has completed once `drain` fires
            mma_commit(drain);
            mbar_wait(drain, 0, a.err, ERR_TIMEOUT_MMA);
        }
    } else {
        // ---------------- epilogue groups ----------------
        // The scores are read in the 16x256b shape: a thread holds columns
        // 8i + 2(lane%4) + {0, 1} (i = 0..15) of the four rows
        // 32*quarter + lane/4 + 8k (k = 0..3), so that each bias value it
        // loads serves four rows, and keeps a running (max, sum) per row over
        // its own columns; the four threads sharing a row merge at the end.
        const int grp = (warp - 2) / kEpiWarps;
        const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
        const float ks = *a.kscale;
        const uint64_t ks2 = pk(ks, ks);
        const uint32_t lofs = (uint32_t)(quarter * 32) << 16;
        const int cpair = 2 * (lane & 3);
        float Mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float Sr[4] = {0.f, 0.f, 0.f, 0.f};
        for (int t = grp; t < ntiles; t += GROUPS) {
            const int b = t & (kTmemBufs - 1);
            const uint32_t ph = (uint32_t)((t >> 2) & 1);
            if (!mbar_wait(&tfull[b], ph, a.err, ERR_TIMEOUT_EPILOGUE)) break;
            tc_fence_after();
            // v[64 h + 4i + {0,1}]: row k = 2h, v[64 h + 4i + {2,3}]: row k = 2h + 1
            float v[2 * 64];
            tmem_ld16x128(tmem + (uint32_t)(b * BN) + lofs, v);
            tmem_ld16x128(tmem + (uint32_t)(b * BN) + lofs + (16u << 16), v + 64);
            tmem_wait_ld();
            tmem_reg_fence(v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
            const int bs = t % kBiasSlots;
            if (!mbar_wait(&bfull[bs], (uint32_t)((t / kBiasSlots) & 1), a.err,
                           ERR_TIMEOUT_EPILOGUE))
                break;

            // s = acc kappa' + bias, per-row maxima
            const uint64_t* sb =
                reinterpret_cast<const uint64_t*>(sBias + bs * kBiasBytes + cpair * 4);
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint64_t bp = sb[4 * i];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float* w = v + 64 * h + 4 * i;
                    upk(fma2(pk(w[0], w[1]), ks2, bp), w[0], w[1]);
                    upk(fma2(pk(w[2], w[3]), ks2, bp), w[2], w[3]);
                    mx[2 * h] = max3(mx[2 * h], w[0], w[1]);
                    mx[2 * h + 1] = max3(mx[2 * h + 1], w[2], w[3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bempty[bs]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (mx[k] > Mr[k]) {
                    Sr[k] *= ex2(Mr[k] - mx[k]);
                    Mr[k] = mx[k];
                }
            }
            // S += sum 2^{s - M} (rows still at -inf saw only padding: their
            // terms are 2^{-inf - (-inf)}, so they are masked to zero)
            uint64_t acc[4] = {pk(0.f, 0.f), pk(0.f, 0.f), pk(0.f, 0.f), pk(0.f, 0.f)};
            uint64_t nm[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) nm[k] = pk(-Mr[k], -Mr[k]);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float* w = v + 64 * h + 4 * i;
                    float x0, x1, x2, x3;
                    upk(add2(pk(w[0], w[1]), nm[2 * h]), x0, x1);
                    upk(add2(pk(w[2], w[3]), nm[2 * h + 1]), x2, x3);
                    acc[2 * h] = add2(acc[2 * h], pk(ex2(x0), ex2(x1)));
                    acc[2 * h + 1] = add2(acc[2 * h + 1], pk(ex2(x2), ex2(x3)));
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float s0, s1;
                upk(acc[k], s0, s1);
                if (Mr[k] != -INFINITY) Sr[k] += s0 + s1;
            }
        }
        // the four threads sharing each row merge their (max, sum)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                const float Mo = __shfl_xor_sync(0xffffffffu, Mr[k], o);
                const float So = __shfl_xor_sync(0xffffffffu, Sr[k], o);
                const float Mn = fmaxf(Mr[k], Mo);
                Sr[k] = (Mr[k] == -INFINITY ? 0.f : Sr[k] * ex2(Mr[k] - Mn)) +
                        (Mo == -INFINITY ? 0.f : So * ex2(Mo - Mn));
                Mr[k] = Mn;
            }
        }
        // from here on a thread owns the row 32*quarter + lane/4 + 8(lane%4)
        const int kown = lane & 3;
        const float M = kown == 0 ? Mr[0] : kown == 1 ? Mr[1] : kown == 2 ? Mr[2] : Mr[3];
        const float S = kown == 0 ? Sr[0] : kown == 1 ? Sr[1] : kown == 2 ? Sr[2] : Sr[3];
        const int rloc = quarter * 32 + (lane >> 2) + 8 * kown;
        const int64_t row = rt * BM + rloc;

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
                    a.partial[(int64_t)blockIdx.y * a.nr + row] = make_float2(Mt, St);
                } else {
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

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool QRES>
cudaError_t launch_half_tc_t(const TcHalfArgs& a, int row_tiles, size_t smem, cudaStream_t s) {
    const cudaError_t e = cudaFuncSetAttribute(
        k_half_tc<QRES>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_half_tc<QRES><<<dim3((unsigned)row_tiles, (unsigned)a.splits), kHalfThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_half_tc(const TcHalfArgs& a, int row_tiles, bool qres, cudaStream_t s) {
    // settled iterations: the reference-offset kernel (Q resident, d <= 128)
    if (a.use_ref) {
        if (!qres || a.nch > 2) return cudaErrorInvalidValue;
        return launch_half_ref(a, row_tiles, s);
    }
    const size_t smem = half_smem_bytes(a.nch, qres, a.stages);
    const cudaError_t e = qres ? launch_half_tc_t<true>(a, row_tiles, smem, s)
                               : launch_half_tc_t<false>(a, row_tiles, smem, s);
    count_launch();
    return e;
}

// ---------------------------------------------------------------------------
// Fixup of guarded rows: one warp per listed row.  The row's centred
// coordinates times kappa sit in shared memory; each lane scores columns
// lane, lane + 32, ... in FP32 from the raw, centred coordinates, folds them
// into an online (max, sum), and the lanes merge by shuffles.  The list
// length is read once per block; the last block to finish resets the list.
namespace {
constexpr int kFixBlocks = 64;
constexpr int kFixWarps = 8;
}  // namespace

__global__ void __launch_bounds__(kFixWarps * 32) k_fix_tc(TcFixArgs a) {
    __shared__ float sx[kFixWarps][kFixMaxDim];
    __shared__ float st[kFixMaxDim];
    __shared__ unsigned int s_cnt;
    const int d = a.d;
    for (int k = threadIdx.x; k < d; k += blockDim.x) st[k] = a.shift[k];
    if (threadIdx.x == 0) s_cnt = min(*(volatile unsigned int*)&a.fix_count[0], (unsigned int)a.nr);
    __syncthreads();
    const unsigned int cnt = s_cnt;
    const int wl = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned int warps = gridDim.x * kFixWarps;
    for (unsigned int w = blockIdx.x * kFixWarps + wl; w < cnt; w += warps) {
        const int64_t row = a.fix_list[w];
        for (int k = lane; k < d; k += 32) sx[wl][k] = (a.R[row * d + k] - st[k]) * a.kappa;
        __syncwarp();
        float M = -INFINITY, S = 0.f;
        for (int64_t j = lane; j < a.nc; j += 32) {
            const float* y = a.C + j * d;
            float s = a.cbias[j];
            for (int k = 0; k < d; ++k) s = fmaf(sx[wl][k], y[k] - st[k], s);
            if (s > M) {
                S *= ex2(M - s);
                M = s;
            }
            if (M != -INFINITY) S += ex2(s - M);
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
            a.rbias[row] = a.rlogw2[row] - lse2;
        }
        __syncwarp();
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

cudaError_t launch_fix_tc(const TcFixArgs& a, cudaStream_t s) {
    if (a.d > kFixMaxDim) return cudaErrorInvalidValue;
    k_fix_tc<<<kFixBlocks, kFixWarps * 32, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace fs

// tcgen05 tensor-core path (d > 16).
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU", Method 1
// (Proposition 1: the f-update is a row LSE of the biased dot-product score
// matrix (Q K^T + bias)/eps) and Method 2 (streaming kernels: the n x m
// matrix never reaches HBM; row-stationary traversal, online max/sum-exp,
// fused potential write-back).
//
// GB300 design.  One CTA owns a 128-row tile of Q (row-stationary) and a
// range of 128-column tiles of K.  Warp 0 streams K chunks (128 x 64 fp16,
// 16 KB, pre-swizzled in HBM) into a shared-memory ring with cp.async.bulk;
// warp 1 issues tcgen05.mma (M=128, N=128, K=16 steps) into one of two TMEM
// accumulators; warps 2-5 read the 128x128 fp32 score tile out of TMEM
// (one thread per row), add the column bias and fold it into the row's
// running max and sum of 2^s.  The other TMEM buffer keeps the tensor core
// busy meanwhile.  Operands are fp16 with a power-of-two scale per point
// cloud (11-bit significand, the precision of TF32 at the f16 MMA rate).
#include "fs_tc.cuh"
#include "fs_tc_kernels.cuh"

namespace fs {
namespace tc {

// ---------------------------------------------------------------------------
// preparation

// One warp per point: squared norm of the centred point, log2 of its
// weight, and the running max |coordinate| (as ordered bits, atomicMax).
__global__ void k_stats(const float* __restrict__ P, const float* __restrict__ w, int64_t rows,
                        int d, const float* __restrict__ shift, float* __restrict__ norm,
                        float* __restrict__ logw2, unsigned int* __restrict__ absmax_bits) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float s = 0.f, mx = 0.f;
    const float* p = P + row * d;
    for (int k = lane; k < d; k += 32) {
        const float c = p[k] - shift[k];
        s = fmaf(c, c, s);
        mx = fmaxf(mx, fabsf(c));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
        norm[row] = s;
        logw2[row] = log2f(w[row]);
        atomicMax(absmax_bits, __float_as_uint(mx));
    }
}

// exponent e with max * 2^e in [2^14, 2^15) (0 for an all-zero cloud)
__device__ __forceinline__ int scale_exp(unsigned int bits) {
    const float mx = __uint_as_float(bits);
    if (!(mx > 0.f)) return 0;
    int E;
    frexpf(mx, &E);
    return 15 - E;
}

// params[0] = 2^ex, params[1] = 2^ey, params[2] = kappa 2^-(ex+ey)
__global__ void k_scales(const unsigned int* __restrict__ absmax_bits, float kappa,
                         float* __restrict__ params) {
    const int ex = scale_exp(absmax_bits[0]);
    const int ey = scale_exp(absmax_bits[1]);
    params[0] = ldexpf(1.f, ex);
    params[1] = ldexpf(1.f, ey);
    params[2] = ldexpf(kappa, -(ex + ey));
}

// One thread per 16-byte unit (8 fp16) of the tiled, swizzled operand.  If
// `out_lo` is given it receives the rounding remainder fp16(v - fp16(v)), so
// that hi + lo carries about 22 significant bits.
__global__ void k_to_tiles(const float* __restrict__ P, int64_t rows, int d,
                           const float* __restrict__ shift, const float* __restrict__ scale_ptr,
                           int nch, int64_t row_tiles, uint4* __restrict__ out,
                           uint4* __restrict__ out_lo) {
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t units = row_tiles * BM * nch * 8;
    if (unit >= units) return;
    const int u = (int)(unit & 7);
    const int64_t rowc = unit >> 3;            // (tile, chunk, r) flattened with r fastest... see below
    const int r = (int)(rowc % BM);
    const int64_t tc_ = rowc / BM;
    const int chunk = (int)(tc_ % nch);
    const int64_t tile = tc_ / nch;
    const int64_t row = tile * BM + r;
    const float scale = *scale_ptr;
    const int k0 = chunk * BK + u * 8;
    __align__(16) __half h[8];
    __align__(16) __half l[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int k = k0 + q;
        float v = 0.f;
        if (row < rows && k < d) v = (P[row * d + k] - shift[k]) * scale;
        h[q] = __float2half_rn(v);
        l[q] = __float2half_rn(v - __half2float(h[q]));
    }
    const int64_t off = (tile * nch + chunk) * (int64_t)CHUNK_BYTES + swz_offset(r, u * 8);
    *reinterpret_cast<uint4*>(reinterpret_cast<char*>(out) + off) = *reinterpret_cast<const uint4*>(h);
    if (out_lo != nullptr)
        *reinterpret_cast<uint4*>(reinterpret_cast<char*>(out_lo) + off) =
            *reinterpret_cast<const uint4*>(l);
}

// bias[j] = (pot_j - norm_j) L/eps + logw2_j for j < rows, -inf for padding;
// with pot == nullptr the real entries are left alone (only padding is set).
__global__ void k_bias_init(const float* __restrict__ pot, const float* __restrict__ norm,
                            const float* __restrict__ logw2, float l_over_eps, int64_t rows,
                            int64_t rows_pad, float* __restrict__ bias) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= rows_pad) return;
    if (j >= rows) bias[j] = -INFINITY;
    else if (pot != nullptr) bias[j] = (pot[j] - norm[j]) * l_over_eps + logw2[j];
}

cudaError_t launch_prep_side(const float* P, const float* w, int64_t rows, int d,
                             const float* shift, float* norm, float* logw2,
                             unsigned int* absmax_bits, cudaStream_t s) {
    const int64_t threads = rows * 32;
    k_stats<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(P, w, rows, d, shift, norm, logw2,
                                                              absmax_bits);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_scales(const unsigned int* absmax_bits, float kappa, float* params,
                          cudaStream_t s) {
    k_scales<<<1, 1, 0, s>>>(absmax_bits, kappa, params);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_to_tiles(const float* P, int64_t rows, int d, const float* shift,
                            const float* scale_ptr, int nch, int64_t row_tiles, void* out,
                            void* out_lo, cudaStream_t s) {
    const int64_t units = row_tiles * BM * nch * 8;
    k_to_tiles<<<(unsigned)((units + 255) / 256), 256, 0, s>>>(P, rows, d, shift, scale_ptr, nch,
                                                               row_tiles, (uint4*)out,
                                                               (uint4*)out_lo);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_bias_init(const float* pot, const float* norm, const float* logw2,
                             float l_over_eps, int64_t rows, int64_t rows_pad, float* bias,
                             cudaStream_t s) {
    k_bias_init<<<(unsigned)((rows_pad + 255) / 256), 256, 0, s>>>(pot, norm, logw2, l_over_eps,
                                                                   rows, rows_pad, bias);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// half-update

template <bool QRES>
__global__ void __launch_bounds__(kHalfThreads, 1) k_half_tc(TcHalfArgs a) {
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

    constexpr int STAGE_BYTES = QRES ? CHUNK_BYTES : 2 * CHUNK_BYTES;
    uint8_t* sQ = smem;
    uint8_t* sStage = smem + (QRES ? nch * CHUNK_BYTES : 0);
    uint64_t* full = reinterpret_cast<uint64_t*>(sStage + kStages * STAGE_BYTES);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + kTmemBufs;
    uint64_t* qfull = tempty + kTmemBufs;
    uint64_t* drain = qfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < kTmemBufs; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
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
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int t = 0; t < ntiles && ok; ++t) {
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
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA can exit
                int s2 = 0;
                uint32_t ph2 = 0;
                const int skip = issued > kStages ? issued - kStages : 0;
                for (int i = 0; i < issued; ++i) {
                    if (i >= skip) mbar_wait(&full[s2], ph2, a.err, ERR_TIMEOUT_PRODUCER);
                    if (++s2 == kStages) {
                        s2 = 0;
                        ph2 ^= 1u;
                    }
                }
                if (QRES) mbar_wait(qfull, 0, a.err, ERR_TIMEOUT_PRODUCER);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            bool ok = true;
            if (QRES) ok = mbar_wait(qfull, 0, a.err, ERR_TIMEOUT_MMA);
            tc_fence_after();
            int s = 0;
            uint32_t ph = 0;
            for (int t = 0; t < ntiles && ok; ++t) {
                const int b = t % kTmemBufs;
                const uint32_t bph = (uint32_t)((t / kTmemBufs) & 1);
                if (!mbar_wait(&tempty[b], bph ^ 1u, a.err, ERR_TIMEOUT_MMA)) {
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
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16(d_tmem, sdesc_sw128(aaddr + kk * 32), sdesc_sw128(baddr + kk * 32),
                                idesc, (c | kk) != 0);
                    mma_commit(&empty[s]);
                    if (++s == kStages) {
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
        // ---------------- epilogue: one thread per row ----------------
        const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
        const int rloc = quarter * 32 + lane;
        const int64_t row = rt * BM + rloc;
        const float ks = *a.kscale;
        float M = -INFINITY, S = 0.f;
        bool ok = true;
        for (int t = 0; t < ntiles; ++t) {
            const int b = t % kTmemBufs;
            const uint32_t bph = (uint32_t)((t / kTmemBufs) & 1);
            if (!mbar_wait(&tfull[b], bph, a.err, ERR_TIMEOUT_EPILOGUE)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[BN];
            const uint32_t taddr = tmem + (uint32_t)(b * BN) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) tmem_ld32(taddr + q * 32, v + q * 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);

            const float4* bp = reinterpret_cast<const float4*>(a.cbias + (int64_t)(j0 + t) * BN);
            float mx = -INFINITY;
#pragma unroll
            for (int q = 0; q < BN / 4; ++q) {
                const float4 bb = __ldg(bp + q);
                v[4 * q + 0] = fmaf(v[4 * q + 0], ks, bb.x);
                v[4 * q + 1] = fmaf(v[4 * q + 1], ks, bb.y);
                v[4 * q + 2] = fmaf(v[4 * q + 2], ks, bb.z);
                v[4 * q + 3] = fmaf(v[4 * q + 3], ks, bb.w);
                mx = fmaxf(mx, fmaxf(fmaxf(v[4 * q], v[4 * q + 1]), fmaxf(v[4 * q + 2], v[4 * q + 3])));
            }
            if (mx > M) {
                S *= ex2(M - mx);
                M = mx;
            }
            float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
            for (int q = 0; q < BN / 4; ++q) {
                acc0 += ex2(v[4 * q + 0] - M);
                acc1 += ex2(v[4 * q + 1] - M);
                acc2 += ex2(v[4 * q + 2] - M);
                acc3 += ex2(v[4 * q + 3] - M);
            }
            S += (acc0 + acc1) + (acc2 + acc3);
        }
        if (ok && row < a.nr) {
            if (a.splits > 1) {
                a.partial[(int64_t)blockIdx.y * a.nr + row] = make_float2(M, S);
            } else {
                const float lse2 = M + log2f(S);
                if (a.rnorm != nullptr) {
                    a.pot[row] = a.rnorm[row] - a.eps_ln2 * lse2;
                    a.rbias[row] = a.rlogw2[row] - lse2;
                } else {
                    a.pot[row] = lse2;
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

size_t half_smem_bytes(int nch, bool qres) {
    const size_t stage = qres ? CHUNK_BYTES : 2 * CHUNK_BYTES;
    return 1024 /* alignment slack */ + (qres ? (size_t)nch * CHUNK_BYTES : 0) + kStages * stage +
           8 * (2 * kStages + 2 * kTmemBufs + 2) + 16;
}

cudaError_t launch_half_tc(const TcHalfArgs& a, int row_tiles, bool qres, cudaStream_t s) {
    const size_t smem = half_smem_bytes(a.nch, qres);
    dim3 grid((unsigned)row_tiles, (unsigned)a.splits);
    cudaError_t e;
    if (qres) {
        e = cudaFuncSetAttribute(k_half_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        k_half_tc<true><<<grid, kHalfThreads, smem, s>>>(a);
    } else {
        e = cudaFuncSetAttribute(k_half_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        k_half_tc<false><<<grid, kHalfThreads, smem, s>>>(a);
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace fs

// Plan application on the tensor-core path ("FlashSinkhorn: IO-Aware
// Entropic Optimal Transport on GPU", Method 3: barycentric projection and
// gradient as attention-like weighted means, computed by the streaming
// kernels without materialising the plan).
//
// With LSE_i = log2 sum_j 2^{s_ij} from a first streaming pass (the
// half-update kernel in log2-sum-exp mode), the plan row is
//     P_ij = a_i 2^{phi_i + LSE_i} p_ij,   p_ij = 2^{s_ij - LSE_i} in (0, 1],
// phi_i = (f_i - |x~_i|^2) L/eps, so
//     (P V)_i = a_i W_i sum_j p_ij V_j,     W_i = 2^{phi_i + LSE_i}.
// The second pass is FlashAttention-forward shaped: S = Q K^T into TMEM,
// p = 2^{S kappa + beta - LSE} rounded to fp16 into shared memory, and a
// second tcgen05.mma accumulates O += P V_tile in TMEM.  Because every p is
// already normalised by the exact row LSE there is no running-max rescale,
// and split partial sums merge by plain addition.
#include "fs_tc.cuh"

namespace fs {
namespace tc {

// ---------------------------------------------------------------------------
// value preparation

__global__ void k_absmax(const float* __restrict__ V, int64_t len, unsigned int* __restrict__ bits) {
    float mx = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < len;
         i += (int64_t)gridDim.x * blockDim.x)
        mx = fmaxf(mx, fabsf(V[i]));
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) atomicMax(bits, __float_as_uint(mx));
}

__global__ void k_value_scale(const unsigned int* __restrict__ bits, float* __restrict__ params) {
    const float mx = __uint_as_float(bits[0]);
    int e = 0;
    if (mx > 0.f) {
        int E;
        frexpf(mx, &E);
        e = 15 - E;
    }
    params[0] = ldexpf(1.f, e);
    params[1] = ldexpf(1.f, -e);
}

// One thread per 16-byte unit of the transposed value tiles: unit
// (j, kq, n, u) holds V[point j*128 + 64 kq + 8u + q][n] for q = 0..7.
__global__ void k_vt_tiles(const float* __restrict__ V, int64_t m, int k, int kpad,
                           const float* __restrict__ shift, const float* __restrict__ scale_ptr,
                           int64_t col_tiles, uint4* __restrict__ out) {
    const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t units = col_tiles * 2 * (int64_t)kpad * 8;
    if (unit >= units) return;
    const int u = (int)(unit & 7);
    const int64_t rest = unit >> 3;
    const int n = (int)(rest % kpad);
    const int64_t jq = rest / kpad;             // j * 2 + kq
    const int kq = (int)(jq & 1);
    const int64_t j = jq >> 1;
    const float scale = *scale_ptr;
    const float sh = (shift != nullptr && n < k) ? shift[n] : 0.f;
    __align__(16) __half h[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int64_t p = j * BM + kq * 64 + u * 8 + q;
        float v = 0.f;
        if (p < m && n < k) v = (V[p * k + n] - sh) * scale;
        h[q] = __float2half_rn(v);
    }
    // rows of 128 bytes, one per output column n; 8-row swizzle groups
    char* base = reinterpret_cast<char*>(out) + (jq * kpad) * (int64_t)128;
    *reinterpret_cast<uint4*>(base + swz_offset(n, u * 8)) = *reinterpret_cast<const uint4*>(h);
}

cudaError_t launch_absmax(const float* V, int64_t len, unsigned int* bits, cudaStream_t s) {
    int64_t blocks = (len + 255) / 256;
    if (blocks > 2048) blocks = 2048;
    if (blocks < 1) blocks = 1;
    k_absmax<<<(unsigned)blocks, 256, 0, s>>>(V, len, bits);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_value_scale(const unsigned int* bits, float* params, cudaStream_t s) {
    k_value_scale<<<1, 1, 0, s>>>(bits, params);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_vt_tiles(const float* V, int64_t m, int k, int kpad, const float* shift,
                            const float* scale_ptr, int64_t col_tiles, void* out,
                            cudaStream_t s) {
    const int64_t units = col_tiles * 2 * (int64_t)kpad * 8;
    k_vt_tiles<<<(unsigned)((units + 255) / 256), 256, 0, s>>>(V, m, k, kpad, shift, scale_ptr,
                                                               col_tiles, (uint4*)out);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// output of one row from o = sum_j p_ij V~_j (already unscaled) and
// sigma = sum_j p_ij (the same rounded p the tensor core summed).  For V = Y
// the values are centred, y = y~ + t, so sum_j p_ij y_j = o + t sigma.

__device__ __forceinline__ float apply_out(const TcApplyArgs& a, int64_t row, int col, float W,
                                           float o, float sigma) {
    if (a.mode == APPLY_PV || a.mode == APPLY_TAN) return a.a[row] * W * o;
    const float py = o + a.shift[col] * sigma;     // sum_j p_ij y_j
    if (a.mode == APPLY_BARY) return W * py;
    return 2.f * a.a[row] * (a.X[row * (int64_t)a.k + col] - W * py);
}

__global__ void k_merge_apply_tc(TcApplyArgs a) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= a.nr * (int64_t)a.k) return;
    const int64_t row = idx / a.k;
    const int col = (int)(idx - row * a.k);
    const int64_t stride = a.nr * (int64_t)(a.k + 1);
    const int64_t base = row * (a.k + 1);
    float o = 0.f, sigma = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) {
        o += a.partial[sp * stride + base + col];
        sigma += a.partial[sp * stride + base + a.k];
    }
    const float W = exp2f(a.phi[row] + a.lse2[row]);
    a.out[idx] = apply_out(a, row, col, W, o, sigma);
    if (a.mode == APPLY_TAN && col == 0) a.out2[row] = a.a[row] * W * sigma;
}

cudaError_t launch_merge_apply_tc(const TcApplyArgs& a, cudaStream_t s) {
    const int64_t total = a.nr * (int64_t)a.k;
    k_merge_apply_tc<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// the streaming P V kernel
//
// grid = (row tiles, value-column blocks of 128, splits of the column tiles)
// warp 0: producer (K/Q chunk pairs into a 3-deep ring, value tiles into 2 slots)
// warp 1: MMA issuer (S_{t+1} = Q K_{t+1}^T is issued before O += P_t V_t)
// warps 2-5: epilogue, one thread per row
// TAN (APPLY_TAN): every tile also forms T = U K^T in TMEM columns 128..255
// (the ring carries, per tile, the nch (K, Q) chunk sets and then nch (K, U)
// sets); S and T are single-buffered, and p_ij t_ij replaces p_ij.

namespace {
constexpr int kStageA = 4 * CHUNK_BYTES;          // K hi, K lo, Q hi, Q lo
constexpr int kOCol = 2 * BN;                     // TMEM column of the O accumulator
// value-tile slots: KV output rows x 2 halves x 128 B each
__host__ __device__ constexpr int vt_slot_bytes(int kv) { return kv * 2 * 128; }
__host__ __device__ constexpr int vt_slots(int kv) { return kv == 256 ? 1 : 2; }
}  // namespace

// KV output columns per CTA.  With one value slot (KV = 256) the value tile
// of tile t is loaded while the scores of tile t + 1 stream (after its first
// half of chunks), which the MMA thread consumes only after those scores.
template <int KV, bool TAN>
__global__ void __launch_bounds__(kApplyThreads, 1) k_apply_tc(TcApplyArgs a) {
    constexpr int kVtSlot = vt_slot_bytes(KV);
    constexpr int VS = vt_slots(KV);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rt = blockIdx.x;
    const int n0 = blockIdx.y * KV;
    const int kvN = min(KV, a.kpad - n0);             // multiple of 16
    const int j0 = blockIdx.z * a.tiles_per_split;
    const int j1 = min(a.col_tiles, j0 + a.tiles_per_split);
    const int ntiles = j1 - j0;
    const int nch = a.nch;
    const int nent = TAN ? 2 * nch : nch;   // ring entries per tile

    uint8_t* sStage = smem;
    uint8_t* sVT = sStage + kApplyStages * kStageA;
    uint8_t* sP = sVT + VS * kVtSlot;
    uint64_t* full = reinterpret_cast<uint64_t*>(sP + 2 * CHUNK_BYTES);
    uint64_t* empty = full + kApplyStages;
    uint64_t* tfull = empty + kApplyStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* vfull = tempty + 2;
    uint64_t* vempty = vfull + 2;
    uint64_t* pfull = vempty + 2;
    uint64_t* pempty = pfull + 1;
    uint64_t* ofull = pempty + 1;
    uint64_t* drain = ofull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kApplyStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
            mbar_init(&vfull[b], 1);
            mbar_init(&vempty[b], 1);
        }
        mbar_init(pfull, kEpiWarps);
        mbar_init(pempty, 1);
        mbar_init(ofull, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kApplyTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            const int64_t qoff = rt * nch * (int64_t)CHUNK_BYTES;
            const char* Qg = reinterpret_cast<const char*>(a.Q) + qoff;
            const char* Qlg = reinterpret_cast<const char*>(a.Qlo) + qoff;
            const char* Ug = TAN ? reinterpret_cast<const char*>(a.U) + qoff : nullptr;
            const char* Ulg = TAN ? reinterpret_cast<const char*>(a.Ulo) + qoff : nullptr;
            const char* VTg = reinterpret_cast<const char*>(a.VT);
            int s = 0, issued = 0, vissued = 0;
            uint32_t ph = 0;
            bool ok = true;
            // value tile of tile t into slot t % VS (its u-th use, u = t / VS)
            auto load_v = [&](int t) -> bool {
                const int vb = t % VS;
                const int u = t / VS;
                if (!mbar_wait(&vempty[vb], (uint32_t)(u & 1) ^ 1u, a.err, ERR_TIMEOUT_PRODUCER))
                    return false;
                const uint32_t vbytes = (uint32_t)kvN * 128u;
                const int64_t j = j0 + t;
                mbar_arrive_expect_tx(&vfull[vb], 2 * vbytes);
                for (int kq = 0; kq < 2; ++kq)
                    bulk_g2s(sVT + vb * kVtSlot + kq * vbytes,
                             VTg + ((j * 2 + kq) * a.kpad + n0) * (int64_t)128, vbytes, &vfull[vb]);
                ++vissued;
                return true;
            };
            for (int t = 0; t < ntiles && ok; ++t) {
                const int64_t j = j0 + t;
                const int64_t koff = j * nch * (int64_t)CHUNK_BYTES;
                const char* Kg = reinterpret_cast<const char*>(a.K) + koff;
                const char* Klg = reinterpret_cast<const char*>(a.Klo) + koff;
                for (int e = 0; e < nent; ++e) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, a.err, ERR_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    const int c = e < nch ? e : e - nch;
                    const bool tpart = TAN && e >= nch;     // (K, U) instead of (K, Q)
                    uint8_t* st = sStage + s * kStageA;
                    const int64_t co = c * (int64_t)CHUNK_BYTES;
                    mbar_arrive_expect_tx(&full[s], kStageA);
                    bulk_g2s(st, Kg + co, CHUNK_BYTES, &full[s]);
                    bulk_g2s(st + CHUNK_BYTES, Klg + co, CHUNK_BYTES, &full[s]);
                    bulk_g2s(st + 2 * CHUNK_BYTES, (tpart ? Ug : Qg) + co, CHUNK_BYTES, &full[s]);
                    bulk_g2s(st + 3 * CHUNK_BYTES, (tpart ? Ulg : Qlg) + co, CHUNK_BYTES, &full[s]);
                    ++issued;
                    if (++s == kApplyStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (VS == 1 && e == nch / 2 && t > 0 && !(ok = load_v(t - 1))) break;
                }
                if (!ok) break;
                if (VS == 2 && !(ok = load_v(t))) break;
            }
            if (ok && VS == 1 && ntiles > 0) ok = load_v(ntiles - 1);
            if (!ok) {
                // let every copy already issued land before the CTA can exit
                int s2 = 0;
                uint32_t ph2 = 0;
                const int skip = issued > kApplyStages ? issued - kApplyStages : 0;
                for (int i = 0; i < issued; ++i) {
                    if (i >= skip) mbar_wait(&full[s2], ph2, a.err, ERR_TIMEOUT_PRODUCER);
                    if (++s2 == kApplyStages) {
                        s2 = 0;
                        ph2 ^= 1u;
                    }
                }
                for (int i = vissued > VS ? vissued - VS : 0; i < vissued; ++i)
                    mbar_wait(&vfull[i % VS], (uint32_t)((i / VS) & 1), a.err, ERR_TIMEOUT_PRODUCER);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idescS = idesc_f16_f32(BM, BN);
            const uint64_t stage_desc0 = sdesc_sw128(smem_u32(sStage));
            const uint64_t p_desc0 = sdesc_sw128(smem_u32(sP));
            const uint64_t vt_desc0 = sdesc_sw128(smem_u32(sVT));
            const uint32_t idescO = idesc_f16_f32(BM, kvN);
            int s = 0;
            uint32_t ph = 0;
            auto issue_S = [&](int t) -> bool {
                // TAN: one S buffer (columns 0..127) and one T buffer (128..255)
                const int b = TAN ? 0 : (t & 1);
                const uint32_t tph = TAN ? (uint32_t)(t & 1) : (uint32_t)((t >> 1) & 1);
                if (!mbar_wait(&tempty[b], tph ^ 1u, a.err, ERR_TIMEOUT_MMA))
                    return false;
                tc_fence_after();
                for (int e = 0; e < nent; ++e) {
                    const int c = e < nch ? e : e - nch;
                    const uint32_t d_tmem = tmem + (uint32_t)((e < nch ? b : 1) * BN);
                    if (!mbar_wait(&full[s], ph, a.err, ERR_TIMEOUT_MMA)) return false;
                    tc_fence_after();
                    // descriptors: the start-address field counts 16-byte units, so a
                    // 32-byte K step is + 2 and a chunk + CHUNK_BYTES / 16
                    const uint64_t kh = stage_desc0 + (uint64_t)(s * (kStageA >> 4));
                    const uint64_t kl = kh + (CHUNK_BYTES >> 4);
                    const uint64_t qh = kh + 2 * (CHUNK_BYTES >> 4), ql = kh + 3 * (CHUNK_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t o = 2 * kk;
                        mma_f16(d_tmem, qh + o, kh + o, idescS, (c | kk) != 0);
                        mma_f16(d_tmem, qh + o, kl + o, idescS, 1);
                        mma_f16(d_tmem, ql + o, kh + o, idescS, 1);
                    }
                    mma_commit(&empty[s]);
                    if (++s == kApplyStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                mma_commit(&tfull[b]);
                return true;
            };
            bool ok = ntiles > 0 ? issue_S(0) : true;
            for (int t = 0; t < ntiles && ok; ++t) {
                if (t + 1 < ntiles && !(ok = issue_S(t + 1))) break;
                if (!mbar_wait(pfull, (uint32_t)(t & 1), a.err, ERR_TIMEOUT_MMA) ||
                    !mbar_wait(&vfull[t % VS], (uint32_t)((t / VS) & 1), a.err, ERR_TIMEOUT_MMA)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t vd = vt_desc0 + (uint64_t)((t % VS) * (kVtSlot >> 4));
#pragma unroll
                for (int kq = 0; kq < 2; ++kq)
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16(tmem + kOCol, p_desc0 + (uint64_t)(kq * (CHUNK_BYTES >> 4) + 2 * kk),
                                vd + (uint64_t)(kq * kvN * 8 + 2 * kk), idescO, (t | kq | kk) != 0);
                mma_commit(pempty);
                mma_commit(&vempty[t % VS]);
            }
            mma_commit(ofull);
            mma_commit(drain);
            mbar_wait(drain, 0, a.err, ERR_TIMEOUT_MMA);
        }
    } else {
        const int quarter = warp & 3;
        const int rloc = quarter * 32 + lane;
        const int64_t row = rt * BM + rloc;
        const bool live = row < a.nr;
        const int64_t rowc = live ? row : a.nr - 1;
        const float ks = *a.kscale;
        const float L = a.lse2[rowc];
        const uint32_t lofs = (uint32_t)(quarter * 32) << 16;
        float sigma = 0.f;
        bool ok = true;
        float tmul = 0.f, tc = 0.f;
        if (TAN) {
            tmul = a.tparams[0];
            tc = -a.crow[rowc] * a.tparams[1];
        }
        for (int t = 0; t < ntiles && TAN; ++t) {
            // S and T of tile t (single buffer), a 32-column quarter at a time
            if (!mbar_wait(&tfull[0], (uint32_t)(t & 1), a.err, ERR_TIMEOUT_EPILOGUE) ||
                !mbar_wait(pempty, (uint32_t)(t & 1) ^ 1u, a.err, ERR_TIMEOUT_EPILOGUE)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float4* bp = reinterpret_cast<const float4*>(a.cbias + (int64_t)(j0 + t) * BN);
#pragma unroll 1
            for (int qq = 0; qq < BN / 32; ++qq) {
                float v[32], tv[32];
                tmem_ld32(tmem + lofs + qq * 32, v);
                tmem_ld32(tmem + (uint32_t)BN + lofs + qq * 32, tv);
                tmem_wait_ld();
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    const int u16 = qq * 4 + g8;
                    const float4 b0 = __ldg(bp + 2 * u16);
                    const float4 b1 = __ldg(bp + 2 * u16 + 1);
                    const float* w = v + 8 * g8;
                    const float* tw = tv + 8 * g8;
                    const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                    float p[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        p[e] = ex2(fmaf(w[e], ks, bb[e]) - L) * fmaf(tw[e], tmul, tc);
                    __align__(16) __half2 h[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        h[q] = live ? __floats2half2_rn(p[2 * q], p[2 * q + 1])
                                    : __floats2half2_rn(0.f, 0.f);
                        const float2 r = __half22float2(h[q]);
                        sigma += r.x + r.y;
                    }
                    const int kq = u16 >> 3, u = u16 & 7;
                    *reinterpret_cast<uint4*>(sP + kq * CHUNK_BYTES + swz_offset(rloc, u * 8)) =
                        *reinterpret_cast<const uint4*>(h);
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&tempty[0]);
                mbar_arrive(pfull);
            }
        }
        for (int t = 0; t < ntiles && !TAN; ++t) {
            const int b = t & 1;
            if (!mbar_wait(&tfull[b], (uint32_t)((t >> 1) & 1), a.err, ERR_TIMEOUT_EPILOGUE)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[BN];
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) tmem_ld32(tmem + (uint32_t)(b * BN) + lofs + q * 32, v + q * 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
            // the P buffer is free once the previous tile's P V has completed
            if (!mbar_wait(pempty, (uint32_t)(t & 1) ^ 1u, a.err, ERR_TIMEOUT_EPILOGUE)) {
                ok = false;
                break;
            }
            const float4* bp = reinterpret_cast<const float4*>(a.cbias + (int64_t)(j0 + t) * BN);
#pragma unroll
            for (int u16 = 0; u16 < BN / 8; ++u16) {
                const float4 b0 = __ldg(bp + 2 * u16);
                const float4 b1 = __ldg(bp + 2 * u16 + 1);
                const float* w = v + 8 * u16;
                float p[8];
                p[0] = ex2(fmaf(w[0], ks, b0.x) - L);
                p[1] = ex2(fmaf(w[1], ks, b0.y) - L);
                p[2] = ex2(fmaf(w[2], ks, b0.z) - L);
                p[3] = ex2(fmaf(w[3], ks, b0.w) - L);
                p[4] = ex2(fmaf(w[4], ks, b1.x) - L);
                p[5] = ex2(fmaf(w[5], ks, b1.y) - L);
                p[6] = ex2(fmaf(w[6], ks, b1.z) - L);
                p[7] = ex2(fmaf(w[7], ks, b1.w) - L);
                __align__(16) __half2 h[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    h[q] = live ? __floats2half2_rn(p[2 * q], p[2 * q + 1]) : __floats2half2_rn(0.f, 0.f);
                    const float2 r = __half22float2(h[q]);
                    sigma += r.x + r.y;
                }
                const int kq = u16 >> 3, u = u16 & 7;
                *reinterpret_cast<uint4*>(sP + kq * CHUNK_BYTES + swz_offset(rloc, u * 8)) =
                    *reinterpret_cast<const uint4*>(h);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull);
        }
        if (mbar_wait(ofull, 0, a.err, ERR_TIMEOUT_EPILOGUE) && ok) {
            tc_fence_after();
            // TAN: the plan entries carried a factor 2^et
            const float unt = TAN ? a.tparams[2] : 1.f;
            const float vinv = *a.vinv * unt;
            sigma *= unt;
            const float W = exp2f(a.phi[rowc] + L);
            float* prow = a.splits > 1
                              ? a.partial + ((int64_t)blockIdx.z * a.nr + row) * (a.k + 1)
                              : nullptr;
            if (live && a.splits > 1 && blockIdx.y == 0) prow[a.k] = sigma;
            if (TAN && live && a.splits == 1 && blockIdx.y == 0) a.out2[row] = a.a[row] * W * sigma;
            for (int q = 0; q < (kvN + 31) / 32; ++q) {
                float o[32];
                tmem_ld32(tmem + kOCol + lofs + q * 32, o);
                tmem_wait_ld();
                if (!live) continue;
                for (int cc = 0; cc < 32; ++cc) {
                    const int col = n0 + q * 32 + cc;
                    if (q * 32 + cc >= kvN || col >= a.k) break;
                    const float ov = o[cc] * vinv;
                    if (a.splits > 1)
                        prow[col] = ov;
                    else
                        a.out[row * (int64_t)a.k + col] = apply_out(a, row, col, W, ov, sigma);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kApplyTmemCols);
    }
}

constexpr size_t apply_smem_bytes(int kv) {
    return 1024 + (size_t)kApplyStages * kStageA + (size_t)vt_slots(kv) * vt_slot_bytes(kv) +
           2 * (size_t)CHUNK_BYTES + 8 * (2 * kApplyStages + 8 + 4) + 16;
}
static_assert(apply_smem_bytes(128) <= kSmemLimit && apply_smem_bytes(256) <= kSmemLimit,
              "plan application does not fit in shared memory");

template <int KV, bool TAN>
cudaError_t launch_apply_kv(const TcApplyArgs& a, int row_tiles, cudaStream_t s) {
    constexpr size_t smem = apply_smem_bytes(KV);
    cudaError_t e = cudaFuncSetAttribute(k_apply_tc<KV, TAN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)row_tiles, (unsigned)((a.kpad + KV - 1) / KV), (unsigned)a.splits);
    k_apply_tc<KV, TAN><<<grid, kApplyThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_apply_tc(const TcApplyArgs& a, int row_tiles, cudaStream_t s) {
    const bool wide = apply_kv(a.nch, a.kpad) == 256;
    cudaError_t e;
    if (a.mode == APPLY_TAN)
        e = wide ? launch_apply_kv<256, true>(a, row_tiles, s) : launch_apply_kv<128, true>(a, row_tiles, s);
    else
        e = wide ? launch_apply_kv<256, false>(a, row_tiles, s) : launch_apply_kv<128, false>(a, row_tiles, s);
    count_launch();
    return e;
}

}  // namespace tc
}  // namespace fs
